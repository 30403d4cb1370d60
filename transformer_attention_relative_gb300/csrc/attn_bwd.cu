// attn_bwd.cu -- backward of the T5-bias relative-position attention, sm_103a.
//
// The forward ("Relative Position Embeddings, in depth", section "T5: one
// scalar per head, looked up by bucket") is, per (batch, head),
//   S = Q K^T / sqrt(d) + bias[bucket(j - p_i), h]  (masked), P = softmax_row(S), O = P V.
// The chain rule gives
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D)  with D_i = sum_j P_ij dP_ij,
//   dQ = dS K / sqrt(d),  dK = dS^T Q / sqrt(d),
//   dbias[b, h] = the sum of dS_ij over every (batch, i, j) whose offset falls
//   in bucket b (the table is learned and every offset of a bucket shares its
//   value: "T5 Relative-Position Bias").
//
// Two kernels, one CTA of four warps per 128-row tile; thread t owns TMEM lane t.
//   relpos_bwd_dq_kernel    one query tile. Two passes over the visible K / V
//                           tiles, each computing S = Q K^T and dP = dO V^T into
//                           TMEM. Pass 1 keeps, per row, the running maximum,
//                           sum and P-weighted sum of dP: the log-sum-exp and D
//                           (D straight from its definition, exact to fp32, so
//                           every row's dS sums to zero and nothing leaks into
//                           the saturated buckets' gradients). Pass 2 forms dS
//                           in registers, writes it (bf16) back to TMEM and
//                           accumulates dQ += dS K with A read from TMEM. It
//                           writes the row statistics for the second kernel and
//                           adds its dS to dbias (per offset in shared memory,
//                           then per bucket).
//   relpos_bwd_dkdv_kernel  one key tile against the query tiles that see it:
//                           S^T = K Q^T and dP^T = V dO^T, P^T and dS^T (bf16)
//                           into TMEM, dV += P^T dO and dK += dS^T Q.
// Every product has a shape of the forward's: the score-type products take two
// K-major 128 x 64 tiles, the accumulating ones take A from TMEM and an
// MN-major 128 x 64 tile as B. Streamed tiles pass through a two-stage ring
// filled by TMA. Thread 0 issues the copies and the products; every wait has a
// time limit, after which the kernel records RELPOS_ERR_DEVICE_TIMEOUT and
// winds down (all threads leave the step loop together).
//
// Tensor memory (512 columns): S 0-127, dP 128-255, P (bf16 pairs) 256-319,
// dS (bf16 pairs) 320-383, accumulators 384-447 (dQ, or dV) and 448-511 (dK).

#include <cuda.h>
#include <cuda_bf16.h>

#include <atomic>
#include <cstdint>

#include "ptx.cuh"
#include "relpos_bwd.cuh"
#include "relpos_common.cuh"

namespace relpos {
namespace {

constexpr int kBT = 128;  // rows per tile, queries or keys
constexpr int kBwdThreads = 128;
constexpr int kMaxR = 4096;
constexpr uint32_t kTile = kBT * kHeadDim * 2;  // 16 KB
constexpr uint32_t kOffBars = 6 * kTile;        // six tiles, then the barriers
constexpr uint32_t kOffSlot = kOffBars + 64;
constexpr uint32_t kOffAbort = kOffBars + 68;
constexpr uint32_t kOffAux = kOffBars + 128;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kColS = 0, kColDP = 128, kColP = 256, kColDS = 320, kColAcc0 = 384, kColAcc1 = 448;
// barriers: 0 the resident tiles, 1 / 2 ring stage full, 3 scores done, 4 all products done
enum : int { kBarInit = 0, kBarFull = 1, kBarS = 3, kBarFin = 4, kNumBwdBars = 5 };

constexpr uint32_t kIdScore = idesc_bf16_f32(kBT, kBT, 0, 0);     // both K-major
constexpr uint32_t kIdAcc = idesc_bf16_f32(kBT, kHeadDim, 0, 1);  // A in TMEM, B MN-major

RP_DEVI void bwd_error(int* status) {
  if (status) atomicCAS(status, 0, -4);
}

// D (TMEM, 128 columns) = A B^T over the 64-wide head dimension: A and B are
// 128-row tiles in shared memory, K-major (TMA's 128-byte swizzled rows).
RP_DEVI void mma_scores(uint32_t d, uint32_t a_smem, uint32_t b_smem) {
  const uint64_t da = smem_desc_sw128(a_smem, 16, 1024);
  const uint64_t db = smem_desc_sw128(b_smem, 16, 1024);
#pragma unroll
  for (int kk = 0; kk < kHeadDim / 16; ++kk) umma_bf16_ss(d, da + 2 * kk, db + 2 * kk, kIdScore, kk > 0 ? 1u : 0u);
}

// D (TMEM, 64 columns) (+)= A B: A = 128 x 128 bf16 in TMEM (pairs per
// column), B = a 128-row tile in shared memory read MN-major (its rows are the
// reduction index, its 64 columns the output columns).
RP_DEVI void mma_accum(uint32_t d, uint32_t a_tmem, uint32_t b_smem, bool acc) {
  const uint64_t db = smem_desc_sw128(b_smem, 8192, 1024);
#pragma unroll
  for (int kk = 0; kk < kBT / 16; ++kk)
    umma_bf16_ts(d, a_tmem + kk * 8, db + 128 * kk, kIdAcc, (acc || kk > 0) ? 1u : 0u);
}

// Store one 64-wide fp32 row (two 32-column TMEM loads) times `mul` as bf16.
RP_DEVI void store_row_bf16(__nv_bfloat16* dst, const uint32_t (&a)[32], const uint32_t (&b)[32], float mul) {
  uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
  for (int v = 0; v < 8; ++v) {
    const uint32_t* r = v < 4 ? &a[v * 8] : &b[(v - 4) * 8];
    uint32_t w[4];
#pragma unroll
    for (int e = 0; e < 4; ++e)
      w[e] = pack_bf16x2(__uint_as_float(r[2 * e]) * mul, __uint_as_float(r[2 * e + 1]) * mul);
    d4[v] = make_uint4(w[0], w[1], w[2], w[3]);
  }
}

// The bias of every offset in [-R, R] (log2-scaled) for head h; entries 0 and
// 2R serve every offset beyond on their side.
RP_DEVI void build_bias_table(float* tab, const BwdParams& p, int h) {
  for (int x = threadIdx.x; x <= 2 * p.R; x += kBwdThreads)
    tab[x] = __ldg(p.bias + t5_bucket_dev(x - p.R, p.t5) * p.H + h) * kLog2e;
}

// Bounded wait for the copies thread 0 issued and nobody waited on (only on the
// way out after a timeout): the CTA must not exit with a copy in flight.
RP_DEVI void drain_copies(uint32_t sb, bool init_waited, int issued, int consumed) {
  if (!init_waited) mbar_wait(sb + kOffBars + 8u * kBarInit, 0, 100000000ull);
  for (int k = consumed; k < issued; ++k)
    mbar_wait(sb + kOffBars + 8u * (kBarFull + (k & 1)), (k >> 1) & 1, 100000000ull);
}

// ---------------------------------------------------------------- dQ kernel
// Shared memory: tile 0 Q, 1 dO, 2-3 K ring, 4-5 V ring; then the bias table,
// the dS sums per offset and per bucket.
__global__ void __launch_bounds__(kBwdThreads, 1)
    relpos_bwd_dq_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                         const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                         const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sb - raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int bh = blockIdx.y;
  const int h = bh % p.H;
  const int i0 = blockIdx.x * kBT;
  const int R = p.R;
  float* tab = reinterpret_cast<float*>(smem + kOffAux);
  float* hist = tab + (2 * R + 1);   // dS summed per offset in (-R, R)
  float* hist_b = hist + (2 * R + 1);  // per bucket
  volatile int* abort_f = reinterpret_cast<volatile int*>(smem + kOffAbort);
  auto bar = [&](int i) { return sb + kOffBars + 8u * i; };

  const int last_row = min(i0 + kBT, p.Lq) - 1;
  int n_kv = (p.Lk + kBT - 1) / kBT;
  if (p.causal) n_kv = min(n_kv, (last_row + p.q_offset) / kBT + 1);
  const int nsteps = 2 * n_kv;  // pass 1, then pass 2, over the same key tiles

  if (tid == 0) {
    for (int i = 0; i < kNumBwdBars; ++i) mbar_init(bar(i), 1);
    *abort_f = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(sb + kOffSlot, kTmemCols);
    tmem_relinquish();
  }
  build_bias_table(tab, p, h);
  for (int x = tid; x <= 2 * R; x += kBwdThreads) hist[x] = 0.f;
  for (int x = tid; x < p.nb; x += kBwdThreads) hist_b[x] = 0.f;
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffSlot);
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  bool init_waited = false;
  int issued = 0, consumed = 0;  // ring copies issued / waited for (thread 0)
  if (tid == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    mbar_arrive_expect_tx(bar(kBarInit), 2 * kTile);
    tma_load_3d(sb + 0 * kTile, &tmQ, bar(kBarInit), 0, i0, bh);
    tma_load_3d(sb + 1 * kTile, &tmdO, bar(kBarInit), 0, i0, bh);
    mbar_arrive_expect_tx(bar(kBarFull), 2 * kTile);
    tma_load_3d(sb + 2 * kTile, &tmK, bar(kBarFull), 0, 0, bh);
    tma_load_3d(sb + 4 * kTile, &tmV, bar(kBarFull), 0, 0, bh);
    issued = 1;
  }

  const int row = i0 + tid;
  const bool row_ok = row < p.Lq;
  const int prow = row + p.q_offset;
  float m = -INFINITY, l = 0.f, dsum = 0.f, lse2 = 0.f, Drow = 0.f;
  float sumL = 0.f, sumR = 0.f;  // dS of the offsets <= -R and >= R

  for (int s = 0; s < nsteps; ++s) {
    const bool pass2 = s >= n_kv;
    const int kt = pass2 ? s - n_kv : s;
    const int j0 = kt * kBT;
    const int st = s & 1;
    if (tid == 0 && !*abort_f) {
      bool ok = true;
      if (!init_waited) ok = init_waited = mbar_wait(bar(kBarInit), 0);
      if (ok) ok = mbar_wait(bar(kBarFull + st), (s >> 1) & 1);
      if (ok) {
        ++consumed;
        tc_fence_after();
        mma_scores(tmem + kColS, sb + 0 * kTile, sb + (2 + st) * kTile);
        mma_scores(tmem + kColDP, sb + 1 * kTile, sb + (4 + st) * kTile);
        tc_commit(bar(kBarS));
      } else {
        *abort_f = 1;
      }
    }
    if (!mbar_wait(bar(kBarS), s & 1)) *abort_f = 1;
    tc_fence_after();
    // the next step's tiles go to the other stage, whose last readers (the
    // products of step s - 1) completed before the scores of step s
    if (tid == 0 && s + 1 < nsteps && !*abort_f) {
      const int s1 = s + 1, st1 = s1 & 1;
      const int kt1 = s1 >= n_kv ? s1 - n_kv : s1;
      mbar_arrive_expect_tx(bar(kBarFull + st1), 2 * kTile);
      tma_load_3d(sb + (2 + st1) * kTile, &tmK, bar(kBarFull + st1), 0, kt1 * kBT, bh);
      tma_load_3d(sb + (4 + st1) * kTile, &tmV, bar(kBarFull + st1), 0, kt1 * kBT, bh);
      ++issued;
    }
    const int rb = j0 - prow;  // offset of column 0 for this row
#pragma unroll 1
    for (int c0 = 0; c0 < kBT; c0 += 32) {
      uint32_t sr[32], dr[32];
      tmem_ld32(tmem + lane_base + kColS + c0, sr);
      tmem_ld32(tmem + lane_base + kColDP + c0, dr);
      tmem_ld_wait(sr);
      tmem_ld_wait(dr);
      if (!pass2) {
        float x[32];
        float cm = -INFINITY;
#pragma unroll
        for (int e = 0; e < 32; ++e) {
          const int rel = rb + c0 + e;
          const bool valid = row_ok && j0 + c0 + e < p.Lk && (!p.causal || rel <= 0);
          const int idx = min(max(rel + R, 0), 2 * R);
          x[e] = valid ? fmaf(__uint_as_float(sr[e]), p.scale_log2, tab[idx]) : -INFINITY;
          cm = fmaxf(cm, x[e]);
        }
        const float mn = fmaxf(m, cm);
        if (mn != -INFINITY) {
          float acc = 0.f, accd = 0.f;
#pragma unroll
          for (int e = 0; e < 32; ++e) {
            const float w = ex2_approx(x[e] - mn);
            acc += w;
            accd = fmaf(w, __uint_as_float(dr[e]), accd);
          }
          const float rs = ex2_approx(m - mn);
          l = fmaf(l, rs, acc);
          dsum = fmaf(dsum, rs, accd);
          m = mn;
        }
      } else {
        uint32_t pk[16];
#pragma unroll
        for (int e = 0; e < 32; e += 2) {
          float ds2[2];
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const int rel = rb + c0 + e + u;
            const bool valid = row_ok && j0 + c0 + e + u < p.Lk && (!p.causal || rel <= 0);
            const int idx = min(max(rel + R, 0), 2 * R);
            const float s2 = fmaf(__uint_as_float(sr[e + u]), p.scale_log2, tab[idx]);
            const float pv = valid ? ex2_approx(s2 - lse2) : 0.f;
            const float ds = pv * (__uint_as_float(dr[e + u]) - Drow);
            ds2[u] = ds;
            if (valid) {
              if (rel <= -R)
                sumL += ds;
              else if (rel >= R)
                sumR += ds;
              else
                atomicAdd(&hist[rel + R], ds);
            }
          }
          pk[e / 2] = pack_bf16x2(ds2[0], ds2[1]);
        }
        tmem_st16(tmem + lane_base + kColDS + c0 / 2, pk);
      }
    }
    if (pass2) tmem_st_wait();
    if (s == n_kv - 1) {  // end of pass 1: the row statistics
      lse2 = m == -INFINITY ? 0.f : m + log2f(l);
      Drow = m == -INFINITY ? 0.f : dsum / l;
      if (row_ok) {
        p.lse[static_cast<size_t>(bh) * p.Lq + row] = lse2;
        p.Dr[static_cast<size_t>(bh) * p.Lq + row] = Drow;
      }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*abort_f) break;
    if (pass2 && tid == 0) mma_accum(tmem + kColAcc0, tmem + kColDS, sb + (2 + st) * kTile, kt > 0);
  }

  // ---------------------------------------------------------------- epilogue
  if (tid == 0) tc_commit(bar(kBarFin));
  if (!mbar_wait(bar(kBarFin), 0)) *abort_f = 1;
  tc_fence_after();
  {
    uint32_t a[32], b[32];
    tmem_ld32(tmem + lane_base + kColAcc0, a);
    tmem_ld32(tmem + lane_base + kColAcc0 + 32, b);
    tmem_ld_wait(a);
    tmem_ld_wait(b);
    if (row_ok && !*abort_f)
      store_row_bf16(p.dQ + (static_cast<size_t>(bh) * p.Lq + row) * kHeadDim, a, b, p.scale);
  }
  // dbias: the saturated sides per warp, then every offset's sum to its bucket
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    sumL += __shfl_xor_sync(0xffffffffu, sumL, o);
    sumR += __shfl_xor_sync(0xffffffffu, sumR, o);
  }
  if ((tid & 31) == 0) {
    if (sumL != 0.f) atomicAdd(&hist_b[t5_bucket_dev(-R, p.t5)], sumL);
    if (sumR != 0.f) atomicAdd(&hist_b[t5_bucket_dev(R, p.t5)], sumR);
  }
  __syncthreads();
  for (int x = tid; x <= 2 * R; x += kBwdThreads)
    if (hist[x] != 0.f) atomicAdd(&hist_b[t5_bucket_dev(x - R, p.t5)], hist[x]);
  __syncthreads();
  if (!*abort_f)
    for (int x = tid; x < p.nb; x += kBwdThreads)
      if (hist_b[x] != 0.f) atomicAdd(p.dbias + x * p.H + h, hist_b[x]);

  if (tid == 0 && *abort_f) {
    drain_copies(sb, init_waited, issued, consumed);
    bwd_error(p.status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------- dK / dV kernel
// Shared memory: tile 0 K, 1 V, 2-3 Q ring, 4-5 dO ring; then the bias table
// and the row statistics (log-sum-exp, D) of the current query tile, two
// buffers.
__global__ void __launch_bounds__(kBwdThreads, 1)
    relpos_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                           const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sb - raw);
  const int tid = threadIdx.x;
  const int warp = tid >> 5;
  const int bh = blockIdx.y;
  const int h = bh % p.H;
  const int j0 = blockIdx.x * kBT;
  const int R = p.R;
  float* tab = reinterpret_cast<float*>(smem + kOffAux);
  float* lse_s = tab + (2 * R + 1);  // [2][128]
  float* d_s = lse_s + 2 * kBT;      // [2][128]
  volatile int* abort_f = reinterpret_cast<volatile int*>(smem + kOffAbort);
  auto bar = [&](int i) { return sb + kOffBars + 8u * i; };

  // query tiles that see a key of this tile: rows i with i + q_offset >= j0
  const int nqt = (p.Lq + kBT - 1) / kBT;
  int first = 0;
  if (p.causal && j0 - p.q_offset > 0) first = (j0 - p.q_offset) / kBT;
  const int nsteps = nqt > first ? nqt - first : 0;

  if (tid == 0) {
    for (int i = 0; i < kNumBwdBars; ++i) mbar_init(bar(i), 1);
    *abort_f = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(sb + kOffSlot, kTmemCols);
    tmem_relinquish();
  }
  build_bias_table(tab, p, h);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffSlot);
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;

  bool init_waited = nsteps == 0;
  int issued = 0, consumed = 0;
  if (tid == 0 && nsteps > 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmdO);
    mbar_arrive_expect_tx(bar(kBarInit), 2 * kTile);
    tma_load_3d(sb + 0 * kTile, &tmK, bar(kBarInit), 0, j0, bh);
    tma_load_3d(sb + 1 * kTile, &tmV, bar(kBarInit), 0, j0, bh);
    mbar_arrive_expect_tx(bar(kBarFull), 2 * kTile);
    tma_load_3d(sb + 2 * kTile, &tmQ, bar(kBarFull), 0, first * kBT, bh);
    tma_load_3d(sb + 4 * kTile, &tmdO, bar(kBarFull), 0, first * kBT, bh);
    issued = 1;
  }

  const int key = j0 + tid;
  const bool key_ok = key < p.Lk;
  for (int s = 0; s < nsteps; ++s) {
    const int i0 = (first + s) * kBT;
    const int st = s & 1;
    {  // this query tile's statistics (the buffer's last readers were two steps ago)
      const int i = i0 + tid;
      lse_s[st * kBT + tid] = i < p.Lq ? __ldg(p.lse + static_cast<size_t>(bh) * p.Lq + i) : 0.f;
      d_s[st * kBT + tid] = i < p.Lq ? __ldg(p.Dr + static_cast<size_t>(bh) * p.Lq + i) : 0.f;
    }
    if (tid == 0 && !*abort_f) {
      bool ok = true;
      if (!init_waited) ok = init_waited = mbar_wait(bar(kBarInit), 0);
      if (ok) ok = mbar_wait(bar(kBarFull + st), (s >> 1) & 1);
      if (ok) {
        ++consumed;
        tc_fence_after();
        mma_scores(tmem + kColS, sb + 0 * kTile, sb + (2 + st) * kTile);   // S^T = K Q^T
        mma_scores(tmem + kColDP, sb + 1 * kTile, sb + (4 + st) * kTile);  // dP^T = V dO^T
        tc_commit(bar(kBarS));
      } else {
        *abort_f = 1;
      }
    }
    __syncthreads();  // the statistics
    if (!mbar_wait(bar(kBarS), s & 1)) *abort_f = 1;
    tc_fence_after();
    if (tid == 0 && s + 1 < nsteps && !*abort_f) {
      const int st1 = (s + 1) & 1;
      mbar_arrive_expect_tx(bar(kBarFull + st1), 2 * kTile);
      tma_load_3d(sb + (2 + st1) * kTile, &tmQ, bar(kBarFull + st1), 0, i0 + kBT, bh);
      tma_load_3d(sb + (4 + st1) * kTile, &tmdO, bar(kBarFull + st1), 0, i0 + kBT, bh);
      ++issued;
    }
    const int rb = key - i0 - p.q_offset;  // offset of column 0 for this key
    const float* lse_t = lse_s + st * kBT;
    const float* d_t = d_s + st * kBT;
#pragma unroll 1
    for (int c0 = 0; c0 < kBT; c0 += 32) {
      uint32_t sr[32], dr[32];
      tmem_ld32(tmem + lane_base + kColS + c0, sr);
      tmem_ld32(tmem + lane_base + kColDP + c0, dr);
      tmem_ld_wait(sr);
      tmem_ld_wait(dr);
      uint32_t pp[16], pd[16];
#pragma unroll
      for (int e = 0; e < 32; e += 2) {
        float pv2[2], ds2[2];
#pragma unroll
        for (int u = 0; u < 2; ++u) {
          const int c = c0 + e + u;
          const int rel = rb - c;
          const bool valid = i0 + c < p.Lq && (!p.causal || rel <= 0);
          const int idx = min(max(rel + R, 0), 2 * R);
          const float s2 = fmaf(__uint_as_float(sr[e + u]), p.scale_log2, tab[idx]);
          const float pv = valid ? ex2_approx(s2 - lse_t[c]) : 0.f;
          pv2[u] = pv;
          ds2[u] = pv * (__uint_as_float(dr[e + u]) - d_t[c]);
        }
        pp[e / 2] = pack_bf16x2(pv2[0], pv2[1]);
        pd[e / 2] = pack_bf16x2(ds2[0], ds2[1]);
      }
      tmem_st16(tmem + lane_base + kColP + c0 / 2, pp);
      tmem_st16(tmem + lane_base + kColDS + c0 / 2, pd);
    }
    tmem_st_wait();
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (*abort_f) break;
    if (tid == 0) {
      mma_accum(tmem + kColAcc0, tmem + kColP, sb + (4 + st) * kTile, s > 0);   // dV += P^T dO
      mma_accum(tmem + kColAcc1, tmem + kColDS, sb + (2 + st) * kTile, s > 0);  // dK += dS^T Q
    }
  }

  // ---------------------------------------------------------------- epilogue
  if (tid == 0) tc_commit(bar(kBarFin));
  if (!mbar_wait(bar(kBarFin), 0)) *abort_f = 1;
  tc_fence_after();
  __nv_bfloat16* dv_row = p.dV + (static_cast<size_t>(bh) * p.Lk + key) * kHeadDim;
  __nv_bfloat16* dk_row = p.dK + (static_cast<size_t>(bh) * p.Lk + key) * kHeadDim;
  if (nsteps > 0) {
    uint32_t a[32], b[32];
    tmem_ld32(tmem + lane_base + kColAcc0, a);
    tmem_ld32(tmem + lane_base + kColAcc0 + 32, b);
    tmem_ld_wait(a);
    tmem_ld_wait(b);
    if (key_ok && !*abort_f) store_row_bf16(dv_row, a, b, 1.f);
    tmem_ld32(tmem + lane_base + kColAcc1, a);
    tmem_ld32(tmem + lane_base + kColAcc1 + 32, b);
    tmem_ld_wait(a);
    tmem_ld_wait(b);
    if (key_ok && !*abort_f) store_row_bf16(dk_row, a, b, p.scale);
  } else if (key_ok) {  // no query sees this key
    uint4* v4 = reinterpret_cast<uint4*>(dv_row);
    uint4* k4 = reinterpret_cast<uint4*>(dk_row);
#pragma unroll
    for (int v = 0; v < 8; ++v) {
      v4[v] = make_uint4(0, 0, 0, 0);
      k4[v] = make_uint4(0, 0, 0, 0);
    }
  }
  if (tid == 0 && *abort_f) {
    drain_copies(sb, init_waited, issued, consumed);
    bwd_error(p.status);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One CTA per SM: the 512 TMEM columns a CTA allocates are all there are.
uint32_t bwd_smem_bytes(int R) {
  const uint32_t tab = (2u * static_cast<uint32_t>(R) + 1u) * 4u;
  const uint32_t dq_aux = 2u * tab + static_cast<uint32_t>(kMaxT5Buckets) * 4u;
  const uint32_t dkdv_aux = tab + 4u * kBT * 4u;
  const uint32_t need = 1024u + kOffAux + (dq_aux > dkdv_aux ? dq_aux : dkdv_aux);
  constexpr uint32_t kOneCtaPerSm = 120u * 1024u;
  return need > kOneCtaPerSm ? need : kOneCtaPerSm;
}

}  // namespace

int bwd_max_R() { return kMaxR; }

cudaError_t launch_bwd(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const CUtensorMap& tmdO, const BwdParams& p, cudaStream_t stream) {
  if (p.R < 1 || p.R > kMaxR || p.nb > kMaxT5Buckets) return cudaErrorInvalidValue;
  const uint32_t smem = bwd_smem_bytes(p.R);
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  static std::atomic<uint64_t> attr_set{0};
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (!bit || !(attr_set.load() & bit)) {
    const int most = static_cast<int>(bwd_smem_bytes(kMaxR));
    cudaError_t e = cudaFuncSetAttribute(relpos_bwd_dq_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(relpos_bwd_dkdv_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, most);
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  const unsigned BH = static_cast<unsigned>(p.B * p.H);
  relpos_bwd_dq_kernel<<<dim3((p.Lq + kBT - 1) / kBT, BH), kBwdThreads, smem, stream>>>(tmQ, tmK, tmV, tmdO, p);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  relpos_bwd_dkdv_kernel<<<dim3((p.Lk + kBT - 1) / kBT, BH), kBwdThreads, smem, stream>>>(tmQ, tmK, tmV, tmdO, p);
  return cudaGetLastError();
}

}  // namespace relpos
