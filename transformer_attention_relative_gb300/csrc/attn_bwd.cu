// attn_bwd.cu -- backward of the T5-bias, ALiBi, Shaw and DeBERTa
// relative-position attention, sm_103a.
//
// The forward ("Relative Position Embeddings, in depth", sections "T5: one
// scalar per head, looked up by bucket" and "ALiBi and RoPE: the two
// endpoints") is, per (batch, head),
//   S = Q K^T / sqrt(d) + b(j - p_i)  (masked), P = softmax_row(S), O = P V,
// with b the head's bias of the key-minus-query offset: the learned
// bias[bucket(offset), h] (T5) or -slope_h |offset| (ALiBi). The chain rule
// gives
//   dV = P^T dO,  dP = dO V^T,  dS = P * (dP - D)  with D_i = sum_j P_ij dP_ij,
//   dQ = dS K / sqrt(d),  dK = dS^T Q / sqrt(d),
//   dbias[b, h] = the sum of dS_ij over every (batch, i, j) whose offset falls
//   in bucket b (every offset of a bucket shares its value: "T5
//   Relative-Position Bias"), dslope_h = -sum dS_ij |j - p_i|.
// Shaw (section "Shaw et al.") and DeBERTa (section "DeBERTa: disentangled
// content and position") put table rows into the logit (and, Shaw, the
// value); their extra terms are sums of the same dS (Shaw: and P) gathered
// by table row, formed by the kernels below and the Shaw / DeBERTa ones at
// the end of the file.
//
// Three kernels:
//   relpos_bwd_stats_kernel  one 128-row query tile per CTA: lse_i (log2
//     units) and D_i, straight from their definitions over S = Q K^T and
//     dP = dO V^T (so every row's dS sums to zero up to rounding, and nothing
//     leaks into a saturated bucket's gradient). Warp 0 loads (TMA), warp 1
//     issues both products per key tile into one of two TMEM buffers, and two
//     compute warpgroups take the key tiles alternately (thread t = query row
//     t), each keeping running statistics; the two are merged at the end.
//     Shaw: also each row's q . a_K and dO . a_V per clipped offset and its
//     sums of P and dS per offset; DeBERTa: each row's dS beyond the band.
//   relpos_bwd_dkdv_kernel   one 128-key tile per CTA against every query tile
//     that sees it, taken in 64-row halves ("sub-steps"): S^T = K Q_h^T and
//     dP^T = V dO_h^T into the half's TMEM buffer; the half's compute warpgroup
//     (thread t = key t) forms P^T and dS^T = P^T (dP^T - D) in bf16 over the
//     buffer's first 32 columns for dV += P^T dO_h and dK += dS^T Q_h, and dS
//     itself into shared memory (query-major, the A operand of
//     dQ_i = dS K, one product per query tile). A fourth warpgroup adds each
//     dQ_i, scaled, into an fp32 accumulator in global memory. The bias
//     gradient is summed per offset in shared memory (T5) or per thread
//     (ALiBi's slope) and added once per CTA; DeBERTa's band dS is scattered
//     by table row to global memory.
//   relpos_bwd_dq_convert_kernel  the dQ accumulator to bf16.
// Shaw then adds its a_K term to dQ and sums the tables' gradients (final and
// reduce kernels); DeBERTa folds the far sums into its gathered dS and runs
// its four table products as plain GEMMs (cuBLAS).
// Products of one CTA queue on the tensor core while the compute warpgroups
// work on the other buffer. Every wait has a time limit, after which the kernel
// records RELPOS_ERR_DEVICE_TIMEOUT and winds down without hanging.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cublas_v2.h>

#include <atomic>
#include <cstdint>
#include <mutex>

#include "ptx.cuh"
#include "relpos_bwd.cuh"
#include "relpos_common.cuh"

namespace relpos {
namespace {

constexpr int kBT = 128;  // rows per tile, queries or keys
constexpr int kMaxR = 1024;
constexpr int kMaxShawK = 16;  // Shaw backward: the statistics kernel holds 6 x 128 rows of 2k + 2 floats
constexpr uint32_t kTile = kBT * kHeadDim * 2;  // 16 KB
constexpr uint32_t kHalfTile = kTile / 2;       // 64 rows

constexpr uint32_t kIdS128 = idesc_bf16_f32(kBT, kBT, 0, 0);        // S = Q K^T (stats)
constexpr uint32_t kIdS64 = idesc_bf16_f32(kBT, 64, 0, 0);          // S^T = K Q_h^T (64 queries)
constexpr uint32_t kIdAcc = idesc_bf16_f32(kBT, kHeadDim, 0, 1);    // A from TMEM or K-major smem, B MN-major

RP_DEVI void bwd_error(int* status) {
  if (status) atomicCAS(status, 0, -4);
}

// T5 bias tables. A near tile's offsets reach at most 254 beyond the
// saturation distance R on either side (a 128 x 128 tile spans 255 offsets),
// so the extended table E covers offsets -R - kTabPad ... R + kTabPad, entry
// x holding the log2-scaled bias of offset x - R - kTabPad. It is kept as four
// copies shifted by one entry each, so that any run of 64 consecutive
// entries starts 16-byte aligned in one of them and is read with 16-byte
// loads; the copies sit 32 bytes apart modulo 128 (fewer bank conflicts
// between lanes reading different copies). The query-major statistics
// kernel reads E by increasing offset; the key-major dK / dV kernel reads
// it reversed (F[y] = E[n - 1 - y]), so that its offsets also increase with
// the column.
constexpr int kTabPad = 256;
__host__ __device__ inline int tab_len(int R) { return 2 * R + 2 * kTabPad + 1; }
// floats per copy: room for a 64-entry window at the end, and 8 floats
// beyond a multiple of 32 (the 32-byte placement above)
__host__ __device__ inline int tab_stride(int R) { return ((tab_len(R) + 64 + 31) & ~31) + 8; }
// The head's biases per bucket (log2-scaled) into bsm[nb]; the caller
// synchronizes before build_bias_copies reads them.
RP_DEVI void load_bucket_bias(float* bsm, const BwdParams& p, int h, int tid) {
  if (tid < p.nb) bsm[tid] = __ldg(p.bias + tid * p.H + h) * kLog2e;
}
// Copy 0 first (with the bucket of each entry into bk[] when given: bk[y]
// for entry y of E, offset y - R - kTabPad), then, after a named barrier of
// the nthreads callers, copies 1 .. 3 from copy 0; the caller synchronizes
// before reading them.
RP_DEVI void build_bias_copies(float* base, const float* bsm, const BwdParams& p, bool reversed, int tid,
                               int nthreads, int bar_id, uint8_t* bk) {
  const int n = tab_len(p.R), st = tab_stride(p.R);
  for (int e = tid; e < st; e += nthreads) {
    int y = min(e, n - 1);           // entry of F (reversed) or E
    if (reversed) y = n - 1 - y;     // F[y] = E[n - 1 - y]
    const int b = t5_bucket_dev(y - p.R - kTabPad, p.t5);
    base[e] = bsm[b];
    if (bk != nullptr && e < n) bk[y] = static_cast<uint8_t>(b);
  }
  named_bar_sync(bar_id, nthreads);
  for (int x = st + tid; x < 4 * st; x += nthreads) {
    const int k = x / st, e = x - k * st;
    base[x] = base[min(e + k, n - 1)];
  }
}
// the 64 entries from index w of a table kept as four shifted copies
RP_DEVI const float4* tab_window(const float* base, int R, int w) {
  const int k = w & 3;
  return reinterpret_cast<const float4*>(base + k * tab_stride(R) + (w - k));
}

// Tiled bulk reduction shared -> global: element-wise fp32 add of a staged
// box into the tensor (rows past its end are dropped); completion through a
// bulk async-group of the issuing thread.
RP_DEVI void tma_reduce_add_3d(const void* tmap, uint32_t src, int c0, int c1, int c2) {
  asm volatile("cp.reduce.async.bulk.tensor.3d.global.shared::cta.add.tile.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   tmap),
               "r"(src), "r"(c0), "r"(c1), "r"(c2)
               : "memory");
}
RP_DEVI void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// the bulk groups' shared-memory reads are done (the source may be reused)
RP_DEVI void bulk_wait_read() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
RP_DEVI void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// 8 consecutive 32-bit TMEM columns of this thread's lane.
RP_DEVI void tmem_st8(uint32_t taddr, const uint32_t (&r)[8]) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr), "r"(r[0]),
               "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}

// Untiled bulk copy global -> shared (16-byte aligned, size a multiple of 16)
// completing on an mbarrier's transaction count.
RP_DEVI void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
               "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}

RP_DEVI void st_shared_u16(uint32_t addr, uint16_t v) {
  asm volatile("st.shared.u16 [%0], %1;" ::"r"(addr), "h"(v) : "memory");
}
// Predicated shared-memory store without a branch (the lanes disagree).
RP_DEVI void st_shared_f32_if(uint32_t addr, float v, int pred) {
  asm volatile("{\n\t.reg .pred q;\n\tsetp.ne.b32 q, %2, 0;\n\t@q st.shared.f32 [%0], %1;\n\t}" ::"r"(addr), "f"(v),
               "r"(pred)
               : "memory");
}
// Dot product of a row of 64 values with a bf16 table row in shared memory
// (64 values, 128 contiguous bytes; every lane reads the same row).
RP_DEVI float dot64_bf16(const float (&v)[64], const __nv_bfloat16* row) {
  const uint4* r4 = reinterpret_cast<const uint4*>(row);
  float2 acc = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < 8; ++c) {
    const uint4 u = r4[c];
    const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
      acc = __ffma2_rn(make_float2(v[8 * c + 2 * e], v[8 * c + 2 * e + 1]), t, acc);
    }
  }
  return acc.x + acc.y;
}

// DeBERTa: the relative part of the logit (log2 units) of query row i (at
// position pi) and key j at band offset m = j - pi + k: the band value for
// 1 <= m <= 2k - 1, else the row's saturated c2p value plus the key's
// saturated p2c value of that side. i and j are clamped into the arrays
// (the elements outside them are masked).
RP_DEVI float deberta_bias(const BwdParams& p, int bh, int i, int pi, int j, int m) {
  const int ic = min(i, p.Lq - 1), jc = min(j, p.Lk - 1);
  if (m >= 1 && m <= 2 * p.kc - 1) {
    const int sh = (ic + p.q_offset - p.kc) & 7;  // the row's own shift
    const unsigned short u = __ldg(reinterpret_cast<const unsigned short*>(p.band) +
                                   (static_cast<size_t>(bh) * p.Lq + ic) * p.band_pitch + sh + m);
    return __uint_as_float(static_cast<uint32_t>(u) << 16);
  }
  const int side = m >= 2 * p.kc ? 1 : 0;
  (void)pi;
  return __ldg(p.c2p_const + (static_cast<size_t>(bh) * 2 + side) * p.const_pitch + ic) +
         __ldg(p.p2c_ends + (static_cast<size_t>(bh) * 2 + side) * p.ends_pitch + jc);
}

// ================================================================ stats kernel
// 12 warps: 0 TMA producer, 1 MMA issuer (TMEM owner), 2-3 idle, 4-7 and 8-11
// the compute warpgroups of TMEM buffers 0 and 1 (even / odd key tiles).
constexpr int kStThreads = 384;
constexpr uint32_t kStOffQ = 0, kStOffdO = kTile, kStOffRing = 2 * kTile;  // ring: stages x (K, V)
// the ring's depth (4 stages; Shaw, whose tables fill shared memory, 2), the
// barriers and the shared-memory offsets that follow from it
template <int MODE>
struct StLayout {
  static constexpr int kStages = MODE == 1 ? 2 : 4;
  static constexpr uint32_t kOffBar = kStOffRing + kStages * 2 * kTile;
  static constexpr uint32_t kOffAux = kOffBar + 256;
  static constexpr uint32_t kBarQ = 0;
  static constexpr uint32_t kBarFull = 1;                 // + stage
  static constexpr uint32_t kBarEmpty = 1 + kStages;      // + stage
  static constexpr uint32_t kBarS = 1 + 2 * kStages;      // + buffer
  static constexpr uint32_t kBarSFree = 3 + 2 * kStages;  // + buffer
  static constexpr uint32_t kNumBars = 5 + 2 * kStages;
};
constexpr uint32_t kStSlot = 128, kStAbort = 132;

template <int MODE>
__global__ void __launch_bounds__(kStThreads, 1)
    relpos_bwd_stats_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                            const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                            const BwdParams p) {
  using L = StLayout<MODE>;
  constexpr int S = L::kStages;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sb - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.y, h = bh % p.H;
  const int i0 = blockIdx.x * kBT;
  auto bar = [&](uint32_t i) { return sb + L::kOffBar + 8u * i; };
  volatile int* abort_f = reinterpret_cast<volatile int*>(smem + L::kOffBar + kStAbort);
  float* tab = reinterpret_cast<float*>(smem + L::kOffAux);                 // T5: 4 copies of E
  // Shaw: a_K, a_V (bf16, 64 rows of 64), then per row q . a_K and dO . a_V
  // (nr floats), then each warpgroup's sums per clipped offset of P and P dP
  float* shw = tab + (MODE == 0 ? 4 * tab_stride(p.R) : 0);
  float* mrg = shw + (MODE == 1 ? 64 * 64 + 6 * 128 * p.nr : 0);            // [7][128] merge
  float* bsm = mrg + 7 * 128;                                               // T5 bias per bucket

  const int last_row = min(i0 + kBT, p.Lq) - 1;
  int n_kv = (p.Lk + kBT - 1) / kBT;
  if (p.causal) n_kv = min(n_kv, (last_row + p.q_offset) / kBT + 1);

  if (tid == 0) {
    for (uint32_t i = 0; i < L::kNumBars; ++i)
      mbar_init(bar(i), (i == L::kBarSFree || i == L::kBarSFree + 1) ? 128u : 1u);
    *abort_f = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + L::kOffBar + kStSlot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + L::kOffBar + kStSlot);
  griddep_wait();

  // registers: the loading and issuing warps need few, the compute
  // warpgroups hold 64 columns of S and dP at a time (4 x 32 x 56 + 8 x 32 x 224 <= 384 x 168)
  if (warp < 4) {
    setmaxnreg_dec<56>();
  if (warp == 0) {
    // ---------------------------------------------------------- producer
    int issued = 0;
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      tma_prefetch_desc(&tmdO);
      mbar_arrive_expect_tx(bar(L::kBarQ), 2 * kTile);
      tma_load_3d(sb + kStOffQ, &tmQ, bar(L::kBarQ), 0, i0, bh);
      tma_load_3d(sb + kStOffdO, &tmdO, bar(L::kBarQ), 0, i0, bh);
      for (int j = 0; j < n_kv; ++j) {
        const uint32_t st = j % S;
        if (j >= S && !(ok = mbar_wait(bar(L::kBarEmpty + st), ((j / S) - 1) & 1))) break;
        mbar_arrive_expect_tx(bar(L::kBarFull + st), 2 * kTile);
        tma_load_3d(sb + kStOffRing + st * 2 * kTile, &tmK, bar(L::kBarFull + st), 0, j * kBT, bh);
        tma_load_3d(sb + kStOffRing + st * 2 * kTile + kTile, &tmV, bar(L::kBarFull + st), 0, j * kBT, bh);
        ++issued;
      }
      if (!ok) {
        *abort_f = 1;
        bwd_error(p.status);
      }
      // never leave with copies in flight
      mbar_wait(bar(L::kBarQ), 0, 100000000ull);
      for (int j = issued > S ? issued - S : 0; j < issued; ++j)
        mbar_wait(bar(L::kBarFull + (j % S)), (j / S) & 1, 100000000ull);
    }
  } else if (warp == 1) {
    // ---------------------------------------------------------- MMA issuer
    bool ok = mbar_wait_warp(bar(L::kBarQ), 0);
    const uint64_t dq = smem_desc_sw128(sb + kStOffQ, 16, 1024);
    const uint64_t ddo = smem_desc_sw128(sb + kStOffdO, 16, 1024);
    for (int j = 0; ok && j < n_kv; ++j) {
      const uint32_t st = j % S, x = j & 1;
      ok = mbar_wait_warp(bar(L::kBarFull + st), (j / S) & 1);
      if (ok && j >= 2) ok = mbar_wait_warp(bar(L::kBarSFree + x), ((j >> 1) - 1) & 1);
      if (!ok || __any_sync(0xffffffffu, *abort_f != 0)) break;
      tc_fence_after();
      const uint64_t dk = smem_desc_sw128(sb + kStOffRing + st * 2 * kTile, 16, 1024);
      const uint64_t dv = smem_desc_sw128(sb + kStOffRing + st * 2 * kTile + kTile, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk)
        umma_bf16_ss_elect(tmem + x * 256, dq + 2 * kk, dk + 2 * kk, kIdS128, kk > 0 ? 1u : 0u);
#pragma unroll
      for (int kk = 0; kk < kHeadDim / 16; ++kk)
        umma_bf16_ss_elect(tmem + x * 256 + 128, ddo + 2 * kk, dv + 2 * kk, kIdS128, kk > 0 ? 1u : 0u);
      tc_commit_elect(bar(L::kBarS + x));
      tc_commit_elect(bar(L::kBarEmpty + st));
    }
    if (!ok && lane == 0) {
      *abort_f = 1;
      bwd_error(p.status);
    }
  }
  } else {
    setmaxnreg_inc<224>();
    // ---------------------------------------------------------- compute
    // the bias table, built by the warpgroups that read it while the first
    // tiles load and the first products run
    if constexpr (MODE == 0) {
      const int ct = static_cast<int>(threadIdx.x) - 128;  // 0 .. 255
      load_bucket_bias(bsm, p, h, ct);
      named_bar_sync(2, 256);
      build_bias_copies(tab, bsm, p, false, ct, 256, 2, nullptr);
      named_bar_sync(2, 256);
    }
    if constexpr (MODE == 1) {
      // Shaw: the tables, the zeroed per-offset sums, then every row's
      // q . a_K[r] (log2-scaled, warpgroup 0) and dO . a_V[r] (warpgroup 1)
      // for the clipped offsets r, into shared memory and to global memory
      // (the dK / dV kernel reads them), with the saturated ends apart
      const int ct = static_cast<int>(threadIdx.x) - 128;  // 0 .. 255
      const int nrel = 2 * p.kc + 1;
      __nv_bfloat16* aKs = reinterpret_cast<__nv_bfloat16*>(shw);
      __nv_bfloat16* aVs = aKs + 64 * 64;
      for (int i = ct; i < nrel * 8; i += 256) {
        reinterpret_cast<uint4*>(aKs)[i] = __ldg(reinterpret_cast<const uint4*>(p.aK) + i);
        reinterpret_cast<uint4*>(aVs)[i] = __ldg(reinterpret_cast<const uint4*>(p.aV) + i);
      }
      float* bins0 = shw + 64 * 64 + 2 * 128 * p.nr;
      for (int i = ct; i < 4 * 128 * p.nr; i += 256) bins0[i] = 0.f;
      if (!mbar_wait(bar(L::kBarQ), 0)) *abort_f = 1;  // the Q and dO tiles
      named_bar_sync(2, 256);
      const int xx = (warp - 4) >> 2, tt = ((warp & 3) << 5) | lane;
      const uint8_t* tile = smem + (xx == 0 ? kStOffQ : kStOffdO);
      float v[64];
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        const uint4 u = *reinterpret_cast<const uint4*>(tile + tt * 128 + ((c ^ (tt & 7)) << 4));
        const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
          v[8 * c + 2 * e] = f.x;
          v[8 * c + 2 * e + 1] = f.y;
        }
      }
      float* dst = shw + 64 * 64 + (xx * 128 + tt) * p.nr;
      const __nv_bfloat16* tb = xx == 0 ? aKs : aVs;
      const float sc = xx == 0 ? p.scale_log2 : 1.f;
      const size_t grow = static_cast<size_t>(bh) * p.lq_pad + i0 + tt;
      float* g = (xx == 0 ? p.shT : p.shU) + grow * p.nr;
#pragma unroll 1
      for (int r = 0; r < nrel; ++r) {
        const float val = dot64_bf16(v, tb + r * 64) * sc;
        dst[r] = val;
        g[r] = val;
      }
      named_bar_sync(2, 256);
    }
    const int x = (warp - 4) >> 2;  // TMEM buffer / parity of the key tiles taken
    const int t = ((warp & 3) << 5) | lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int row = i0 + t;
    const int prow = row + p.q_offset;
    const int R = p.R;
    float alibi = 0.f;  // ALiBi: slope (log2 units) per unit of distance
    if constexpr (MODE == 3) alibi = __ldg(p.slopes + h) * kLog2e;
    // running row statistics in log2 units: maximum m (raised lazily, by more
    // than kRescale at a time, which bounds every term by 2^kRescale), sum l
    // of 2^(x - m) and dsum of 2^(x - m) dP
    float m = -INFINITY;
    float2 l2 = make_float2(0.f, 0.f), d2 = make_float2(0.f, 0.f);
    const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
    bool err = false;
    int cnt = 0;
    // Shaw: this row's q . a_K and dO . a_V, this warpgroup's sums per
    // clipped offset of P and P dP (the in-band offsets meet one key each; the
    // two ends gather the keys beyond the clip, kept in registers), rescaled
    // with l and dsum
    const float* Trow = MODE == 1 ? shw + 64 * 64 + t * p.nr : nullptr;
    const float* Urow = MODE == 1 ? shw + 64 * 64 + (128 + t) * p.nr : nullptr;
    float* bp_row = MODE == 1 ? shw + 64 * 64 + (2 * 128 + x * 128 + t) * p.nr : nullptr;
    float* bd_row = MODE == 1 ? shw + 64 * 64 + (4 * 128 + x * 128 + t) * p.nr : nullptr;
    float sLl = 0.f, sRl = 0.f, sLd = 0.f, sRd = 0.f;
    for (int j = x; j < n_kv; j += 2, ++cnt) {
      const bool ok = mbar_wait(bar(L::kBarS + x), cnt & 1);
      err = __any_sync(0xffffffffu, !ok);
      // leave together: the TMEM loads below are warp-collective
      if (err || __any_sync(0xffffffffu, *abort_f != 0)) break;
      tc_fence_after();
      const int j0 = j * kBT;
      // tile classes (uniform over the CTA): offsets key - query position
      // run from rel_lo to rel_hi; rows past Lq are not masked (their
      // statistics are never used)
      const int rel_hi = j0 + kBT - 1 - (i0 + p.q_offset), rel_lo = j0 - (i0 + kBT - 1 + p.q_offset);
      const bool nomask = j0 + kBT <= p.Lk && (!p.causal || rel_hi <= 0);
      const bool far_l = (MODE == 0 && rel_hi <= -R) || ((MODE == 1 || MODE == 2) && rel_hi <= -p.kc);
      const bool far_r = (MODE == 0 && p.t5.bidir && rel_lo >= R) || ((MODE == 1 || MODE == 2) && rel_lo >= p.kc);
      // one row constant: T5 beyond the saturation distance, Shaw beyond the
      // clip; ALiBi with every key on one side (the rest is linear in the
      // column); DeBERTa beyond the band (plus each key's saturated p2c
      // value). T5 near tiles without masking read their biases 4 at a time.
      const bool fast = nomask && (MODE != 3 ? (far_l || far_r) : (rel_hi <= 0 || rel_lo >= 0));
      const bool near_t5 = MODE == 0 && nomask && !fast;
#pragma unroll 1
      for (int c0 = 0; c0 < kBT; c0 += 64) {
        uint32_t sr[64], dr[64];
        tmem_ld32(tmem + lane_base + x * 256 + c0, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld32(tmem + lane_base + x * 256 + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_ld32(tmem + lane_base + x * 256 + 128 + c0, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
        tmem_ld32(tmem + lane_base + x * 256 + 128 + c0 + 32, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
        tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
        if (c0 + 64 == kBT) {  // the buffer is read: the products of tile j + 2 may overwrite it
          tc_fence_before();
          mbar_arrive(bar(L::kBarSFree + x));
        }
        float* xv = reinterpret_cast<float*>(sr);
        float bc = 0.f;  // the row constant of a fast tile (log2 units)
        float ue = 0.f;  // Shaw: dO . a_V of the fast tile's side
        float mx;
        if (near_t5) {
          // E index of column c: j0 + c0 + c - prow + R + kTabPad
          const float4* bw = tab_window(tab, R, j0 + c0 - prow + R + kTabPad);
          float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
          for (int q = 0; q < 16; ++q) {
            const float4 b4 = bw[q];
            const float2 a = __ffma2_rn(make_float2(xv[4 * q], xv[4 * q + 1]), sc2, make_float2(b4.x, b4.y));
            const float2 c = __ffma2_rn(make_float2(xv[4 * q + 2], xv[4 * q + 3]), sc2, make_float2(b4.z, b4.w));
            xv[4 * q] = a.x;
            xv[4 * q + 1] = a.y;
            xv[4 * q + 2] = c.x;
            xv[4 * q + 3] = c.y;
            m0 = max3f(m0, a.x, a.y);
            m1 = max3f(m1, c.x, c.y);
          }
          mx = fmaxf(m0, m1);
        } else if (fast) {
          if constexpr (MODE == 0) {
            bc = far_l ? tab[R + kTabPad - R] : tab[R + kTabPad + R];  // biases of offsets -R, R
          } else if constexpr (MODE == 1) {
            bc = Trow[far_l ? 0 : 2 * p.kc];
            ue = Urow[far_l ? 0 : 2 * p.kc];
          } else if constexpr (MODE == 2) {
            const size_t side = far_l ? 0 : 1;
            bc = __ldg(p.c2p_const + (static_cast<size_t>(bh) * 2 + side) * p.const_pitch + min(row, p.Lq - 1));
            const float4* pe =
                reinterpret_cast<const float4*>(p.p2c_ends + (static_cast<size_t>(bh) * 2 + side) * p.ends_pitch + j0 + c0);
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float4 e = __ldg(pe + q);
              const float2 a = __ffma2_rn(make_float2(xv[4 * q], xv[4 * q + 1]), sc2, make_float2(e.x, e.y));
              const float2 b = __ffma2_rn(make_float2(xv[4 * q + 2], xv[4 * q + 3]), sc2, make_float2(e.z, e.w));
              xv[4 * q] = a.x;
              xv[4 * q + 1] = a.y;
              xv[4 * q + 2] = b.x;
              xv[4 * q + 3] = b.y;
            }
          } else {
            // -slope |j - p| = g (j - p) with g = slope (keys behind) or -slope (ahead):
            // scaled scores plus g c, then the row constant g (j0 + c0 - p)
            const float g = rel_hi <= 0 ? alibi : -alibi;
            bc = g * static_cast<float>(j0 + c0 - prow);
            const float2 g2 = make_float2(g, g);
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
              const float2 v = __ffma2_rn(make_float2(static_cast<float>(c), static_cast<float>(c + 1)), g2,
                                          __fmul2_rn(make_float2(xv[c], xv[c + 1]), sc2));
              xv[c] = v.x;
              xv[c + 1] = v.y;
            }
          }
          float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
          for (int c = 0; c < 64; c += 4) {
            m0 = max3f(m0, xv[c], xv[c + 1]);
            m1 = max3f(m1, xv[c + 2], xv[c + 3]);
          }
          mx = MODE <= 1 ? fmaf(fmaxf(m0, m1), p.scale_log2, bc) : fmaxf(m0, m1) + bc;
        } else {
          float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const int rel = j0 + c0 + c - prow;
            const bool valid = (j0 + c0 + c < p.Lk) & (!p.causal | (rel <= 0));
            float b;
            if constexpr (MODE == 0) {
              b = tab[min(max(rel + R + kTabPad, 0), tab_len(R) - 1)];
            } else if constexpr (MODE == 1) {
              b = Trow[min(max(rel, -p.kc), p.kc) + p.kc];  // (U joins dP in the exponential loop)
            } else if constexpr (MODE == 2) {
              b = deberta_bias(p, bh, row, prow, j0 + c0 + c, rel + p.kc);
            } else {
              b = -alibi * fabsf(static_cast<float>(rel));
            }
            xv[c] = valid ? fmaf(xv[c], p.scale_log2, b) : -INFINITY;
            if (c & 1)
              m1 = fmaxf(m1, xv[c]);
            else
              m0 = fmaxf(m0, xv[c]);
          }
          mx = fmaxf(m0, m1);
        }
        // lazy maximum: rescale the sums only when it grows by more than 2^8
        if (mx > m + 8.f) {
          const float a = ex2_approx(m - mx);  // 0 while m = -inf
          l2 = __fmul2_rn(l2, make_float2(a, a));
          d2 = __fmul2_rn(d2, make_float2(a, a));
          if constexpr (MODE == 1 || MODE == 2) {
            sLl *= a;
            sRl *= a;
            sLd *= a;
            sRd *= a;
          }
          if constexpr (MODE == 1) {
#pragma unroll 1
            for (int r = 0; r < 2 * p.kc + 1; ++r) {
              bp_row[r] *= a;
              bd_row[r] *= a;
            }
          }
          m = mx;
        }
        const float mu = m == -INFINITY ? 0.f : m;
        // 2^(x - m): fast tiles scale the raw scores (T5, Shaw) inside the FMA
        const float2 mul2 = (MODE <= 1 && fast) ? sc2 : make_float2(1.f, 1.f);
        const float off = bc - mu;
        const float2 off2 = make_float2(off, off);
        if constexpr (MODE == 1) {
          if (fast) {
            // beyond the clip: dP gains dO . a_V of the side (added once,
            // times the tile's sum of P); the tile's sums go to that side
            float2 tl = make_float2(0.f, 0.f), td = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
              float2 e = __ffma2_rn(make_float2(xv[c], xv[c + 1]), mul2, off2);
              e.x = ex2_approx(e.x);
              e.y = ex2_approx(e.y);
              tl = __fadd2_rn(tl, e);
              td = __ffma2_rn(e, make_float2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])), td);
            }
            const float sl = tl.x + tl.y, sd = fmaf(ue, sl, td.x + td.y);
            l2.x += sl;
            d2.x += sd;
            if (far_l) {
              sLl += sl;
              sLd += sd;
            } else {
              sRl += sl;
              sRd += sd;
            }
          } else {
            // per element: in-band offsets into their (row, offset) entries
            // (one key each), the others to the side sums
            const uint32_t bp_a = smem_u32(bp_row), bd_a = smem_u32(bd_row);
#pragma unroll
            for (int c = 0; c < 64; ++c) {
              const int rel = j0 + c0 + c - prow;
              const int ri = min(max(rel, -p.kc), p.kc) + p.kc;
              const float e = ex2_approx(xv[c] - mu);
              const float dd = e * (__uint_as_float(dr[c]) + Urow[ri]);
              l2.x += e;
              d2.x += dd;
              const int inb = (rel > -p.kc) & (rel < p.kc);
              const uint32_t ra = 4u * static_cast<uint32_t>(ri);
              st_shared_f32_if(bp_a + ra, e, inb);
              st_shared_f32_if(bd_a + ra, dd, inb);
              sLl += rel <= -p.kc ? e : 0.f;
              sLd += rel <= -p.kc ? dd : 0.f;
              sRl += rel >= p.kc ? e : 0.f;
              sRd += rel >= p.kc ? dd : 0.f;
            }
          }
        } else if constexpr (MODE == 2) {
          // DeBERTa: the row's sums over the keys beyond the band on each
          // side (their dS sums feed the saturated table rows)
          if (fast) {
            float2 tl = make_float2(0.f, 0.f), td = make_float2(0.f, 0.f);
#pragma unroll
            for (int c = 0; c < 64; c += 2) {
              float2 e = __fadd2_rn(make_float2(xv[c], xv[c + 1]), off2);
              e.x = ex2_approx(e.x);
              e.y = ex2_approx(e.y);
              tl = __fadd2_rn(tl, e);
              td = __ffma2_rn(e, make_float2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])), td);
            }
            const float sl = tl.x + tl.y, sd = td.x + td.y;
            l2.x += sl;
            d2.x += sd;
            if (far_l) {
              sLl += sl;
              sLd += sd;
            } else {
              sRl += sl;
              sRd += sd;
            }
          } else {
#pragma unroll
          for (int c = 0; c < 64; ++c) {
            const float e = ex2_approx(xv[c] - mu);
            const float dd = e * __uint_as_float(dr[c]);
            l2.x += e;
            d2.x += dd;
            const int rel = j0 + c0 + c - prow;
            sLl += rel <= -p.kc ? e : 0.f;
            sLd += rel <= -p.kc ? dd : 0.f;
            sRl += rel >= p.kc ? e : 0.f;
            sRd += rel >= p.kc ? dd : 0.f;
          }
          }
        } else {
#pragma unroll
          for (int c = 0; c < 64; c += 2) {
            float2 e = __ffma2_rn(make_float2(xv[c], xv[c + 1]), mul2, off2);
            e.x = ex2_approx(e.x);
            e.y = ex2_approx(e.y);
            l2 = __fadd2_rn(l2, e);
            d2 = __ffma2_rn(e, make_float2(__uint_as_float(dr[c]), __uint_as_float(dr[c + 1])), d2);
          }
        }
      }
    }
    const float l = l2.x + l2.y, dsum = d2.x + d2.y;
    if (err) {
      *abort_f = 1;
      bwd_error(p.status);
    }
    // merge the two warpgroups' statistics (buffer 1's into buffer 0's)
    if (x == 1) {
      mrg[t] = m;
      mrg[128 + t] = l;
      mrg[256 + t] = dsum;
      if constexpr (MODE == 1 || MODE == 2) {
        mrg[3 * 128 + t] = sLl;
        mrg[4 * 128 + t] = sRl;
        mrg[5 * 128 + t] = sLd;
        mrg[6 * 128 + t] = sRd;
      }
    }
    named_bar_sync(1, 256);
    if (x == 0 && !*abort_f) {
      const float m1 = mrg[t], l1 = mrg[128 + t], d1 = mrg[256 + t];
      const float M = fmaxf(m, m1);
      float lse = 0.f, D = 0.f, w0 = 0.f, w1 = 0.f;
      if (M != -INFINITY) {
        const float a0 = m == -INFINITY ? 0.f : ex2_approx(m - M);
        const float a1 = m1 == -INFINITY ? 0.f : ex2_approx(m1 - M);
        const float lt = l * a0 + l1 * a1;
        lse = M + log2f(lt);
        D = (dsum * a0 + d1 * a1) / lt;
        w0 = a0 / lt;
        w1 = a1 / lt;
      }
      if constexpr (MODE == 2) {
        // the row's dS summed over the keys beyond the band, each side
        // (zero for rows past Lq)
        if (row >= p.Lq) w0 = w1 = 0.f;
        const float pl = sLl * w0 + mrg[3 * 128 + t] * w1, pr = sRl * w0 + mrg[4 * 128 + t] * w1;
        const float dl = sLd * w0 + mrg[5 * 128 + t] * w1, dq = sRd * w0 + mrg[6 * 128 + t] * w1;
        p.rowfar[(static_cast<size_t>(bh) * 2) * p.lq_pad + row] = fmaf(-D, pl, dl);
        p.rowfar[(static_cast<size_t>(bh) * 2 + 1) * p.lq_pad + row] = fmaf(-D, pr, dq);
        // for the dK / dV kernel's sub-steps beyond the band: lse minus the
        // side's saturated c2p value, and D
        const int rowc = min(row, p.Lq - 1);
        float* ge = p.shEnds + static_cast<size_t>(bh) * 4 * p.lq_pad + row;
        ge[0] = lse - p.c2p_const[static_cast<size_t>(bh) * 2 * p.const_pitch + rowc];
        ge[p.lq_pad] = lse - p.c2p_const[(static_cast<size_t>(bh) * 2 + 1) * p.const_pitch + rowc];
        ge[2 * static_cast<size_t>(p.lq_pad)] = D;
        ge[3 * static_cast<size_t>(p.lq_pad)] = D;
      }
      if constexpr (MODE == 1) {
        // per clipped offset: sum of P and of dS = P (dP - D) over the
        // row's keys at that offset (zero for rows past Lq)
        if (row >= p.Lq) w0 = w1 = 0.f;
        const float* bp1 = shw + 64 * 64 + (3 * 128 + t) * p.nr;
        const float* bd1 = shw + 64 * 64 + (5 * 128 + t) * p.nr;
        const size_t gr = (static_cast<size_t>(bh) * p.lq_pad + row) * p.nr;
        const int kc2 = 2 * p.kc;
        // for the dK / dV kernel's tiles beyond the clip: lse - T and D - U
        // of the two end offsets
        float* ge = p.shEnds + static_cast<size_t>(bh) * 4 * p.lq_pad + row;
        ge[0] = lse - Trow[0];
        ge[p.lq_pad] = lse - Trow[kc2];
        ge[2 * static_cast<size_t>(p.lq_pad)] = D - Urow[0];
        ge[3 * static_cast<size_t>(p.lq_pad)] = D - Urow[kc2];
#pragma unroll 1
        for (int r = 0; r <= kc2; ++r) {
          float sp, sd;
          if (r == 0) {
            sp = sLl * w0 + mrg[3 * 128 + t] * w1;
            sd = sLd * w0 + mrg[5 * 128 + t] * w1;
          } else if (r == kc2) {
            sp = sRl * w0 + mrg[4 * 128 + t] * w1;
            sd = sRd * w0 + mrg[6 * 128 + t] * w1;
          } else {
            sp = bp_row[r] * w0 + bp1[r] * w1;
            sd = bd_row[r] * w0 + bd1[r] * w1;
          }
          p.shBP[gr + r] = sp;
          p.shBdS[gr + r] = fmaf(-D, sp, sd);
        }
      }
      // rows past Lq (zero-filled Q and dO: D = 0) fill the padding that the
      // dK / dV kernel reads whole
      p.lse[static_cast<size_t>(bh) * p.lq_pad + row] = lse;
      p.Dr[static_cast<size_t>(bh) * p.lq_pad + row] = D;
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================ dK / dV kernel
// 16 warps: 0 TMA producer, 1 MMA issuer (TMEM owner), 2-3 idle, 4-7 and 8-11
// the compute warpgroups of query halves 0 and 1, 12-15 the dQ warpgroup.
constexpr int kKvThreads = 512;
constexpr uint32_t kKvOffK = 0, kKvOffV = kTile;
// a ring stage: the query tile's Q and dO, then its 128 lse and 128 D values
constexpr uint32_t kKvStage = 2 * kTile + 1024;
constexpr uint32_t kKvOffRing = 2 * kTile;                    // 2 stages
constexpr uint32_t kKvOffDS = kKvOffRing + 2 * kKvStage;       // 2 buffers x 2 key halves (K-major)
constexpr uint32_t kKvOffBar = kKvOffDS + 4 * kTile;
constexpr uint32_t kKvOffAux = kKvOffBar + 256;
static_assert(kKvStage % 1024 == 0 && kKvOffDS % 1024 == 0, "swizzled tiles start on 1024-byte boundaries");
enum : uint32_t {
  kKvBarKV = 0,
  kKvBarFull = 1,     // + stage: Q_i, dO_i
  kKvBarEmpty = 3,    // + stage
  kKvBarS = 5,        // + buffer: S^T, dP^T in TMEM
  kKvBarP = 7,        // + buffer: P^T, dS^T written (128 arrivals)
  kKvBarXFree = 9,    // + buffer: dV, dK products of the buffer done
  kKvBarDsFree = 11,  // + dS buffer: the dQ tile staged there has been read by its reduction
  kKvBarDqFull = 13,
  kKvBarDqFree = 14,  // 128 arrivals
  kKvBarFin = 15,
  kKvBarDqStage = 16,  // the dQ warpgroup has staged a dQ tile (128 arrivals)
  kKvNumBars = 17,
};
constexpr uint32_t kKvSlot = 192, kKvAbort = 196;
// TMEM columns: S^T buffers 0-63 / 64-127, dP^T 128-191 / 192-255, dV 256,
// dK 320, dQ tile 384. P^T and dS^T (bf16 pairs, 32 columns) overwrite the
// first half of their buffer's S^T and dP^T.
constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 320, kColDQ = 384;

template <int MODE>
__global__ void __launch_bounds__(kKvThreads, 1)
    relpos_bwd_dkdv_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                           const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmdO,
                           const __grid_constant__ CUtensorMap tmAcc, const BwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t sb = (raw + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sb - raw);
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int bh = blockIdx.y, h = bh % p.H;
  const int j0 = blockIdx.x * kBT;
  const int R = p.R;
  auto bar = [&](uint32_t i) { return sb + kKvOffBar + 8u * i; };
  volatile int* abort_f = reinterpret_cast<volatile int*>(smem + kKvOffBar + kKvAbort);
  // T5: 4 copies of F (the reversed extended bias table); dS summed per
  // offset over the near tiles (entry = E index of the offset); per bucket
  // Shaw: per ring stage, the query tile's lse - T and D - U of the two end
  // offsets (DeBERTa: lse minus the saturated c2p values of the two sides,
  // and D twice)
  float* tab = reinterpret_cast<float*>(smem + kKvOffAux);
  float* hist = tab + (MODE == 0 ? 4 * tab_stride(R) : (MODE == 1 || MODE == 2) ? 2 * 512 : 0);
  float* hist_b = hist + (MODE == 0 ? tab_len(R) : 0);
  float* red = hist_b + kMaxT5Buckets;  // side sums / ALiBi slope partials
  float* bsm = red + 16;                // T5 bias per bucket
  float* strip = bsm + kMaxT5Buckets;   // T5: per compute warp, its sub-step's per-offset sums
  uint8_t* bk = reinterpret_cast<uint8_t*>(strip + 8 * 96);  // T5: bucket of each offset (hist index)

  // query tiles that see a key of this tile: rows i with i + q_offset >= j0
  const int nqt = (p.Lq + kBT - 1) / kBT;
  int first = 0;
  if (p.causal && j0 - p.q_offset > 0) first = (j0 - p.q_offset) / kBT;
  const int ntiles = nqt > first ? nqt - first : 0;
  const int nsub = 2 * ntiles;

  if (tid == 0) {
    for (uint32_t i = 0; i < kKvNumBars; ++i) {
      uint32_t c = 1;
      if (i == kKvBarP || i == kKvBarP + 1 || i == kKvBarDqFree || i == kKvBarDqStage) c = 128;
      mbar_init(bar(i), c);
    }
    *abort_f = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sb + kKvOffBar + kKvSlot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kKvOffBar + kKvSlot);
  griddep_wait();

  if (warp < 4) {
    setmaxnreg_dec<56>();
    if (warp == 0) {
      // -------------------------------------------------------- producer
      if (lane == 0 && ntiles > 0) {
        bool ok = true;
        int issued = 0;
        tma_prefetch_desc(&tmQ);
        tma_prefetch_desc(&tmK);
        tma_prefetch_desc(&tmV);
        tma_prefetch_desc(&tmdO);
        mbar_arrive_expect_tx(bar(kKvBarKV), 2 * kTile);
        tma_load_3d(sb + kKvOffK, &tmK, bar(kKvBarKV), 0, j0, bh);
        tma_load_3d(sb + kKvOffV, &tmV, bar(kKvBarKV), 0, j0, bh);
        for (int i = 0; i < ntiles; ++i) {
          const uint32_t st = i & 1;
          if (i >= 2 && !(ok = mbar_wait(bar(kKvBarEmpty + st), ((i >> 1) - 1) & 1))) break;
          const int q0 = (first + i) * kBT;
          const uint32_t dst = sb + kKvOffRing + st * kKvStage;
          const size_t so = static_cast<size_t>(bh) * p.lq_pad + q0;  // 512-byte aligned rows
          mbar_arrive_expect_tx(bar(kKvBarFull + st), 2 * kTile + 1024 + ((MODE == 1 || MODE == 2) ? 2048 : 0));
          tma_load_3d(dst, &tmQ, bar(kKvBarFull + st), 0, q0, bh);
          tma_load_3d(dst + kTile, &tmdO, bar(kKvBarFull + st), 0, q0, bh);
          bulk_load(dst + 2 * kTile, p.lse + so, 512, bar(kKvBarFull + st));
          bulk_load(dst + 2 * kTile + 512, p.Dr + so, 512, bar(kKvBarFull + st));
          if constexpr (MODE == 1 || MODE == 2) {
#pragma unroll
            for (int e = 0; e < 4; ++e)
              bulk_load(smem_u32(tab) + st * 2048u + e * 512u,
                        p.shEnds + (static_cast<size_t>(bh) * 4 + e) * p.lq_pad + q0, 512, bar(kKvBarFull + st));
          }
          ++issued;
        }
        if (!ok) {
          *abort_f = 1;
          bwd_error(p.status);
        }
        mbar_wait(bar(kKvBarKV), 0, 100000000ull);
        for (int i = issued > 2 ? issued - 2 : 0; i < issued; ++i)
          mbar_wait(bar(kKvBarFull + (i & 1)), (i >> 1) & 1, 100000000ull);
      }
    } else if (warp == 1) {
      // -------------------------------------------------------- MMA issuer
      bool ok = ntiles == 0 || mbar_wait_warp(bar(kKvBarKV), 0);
      const uint64_t dk_a = smem_desc_sw128(sb + kKvOffK, 16, 1024);    // K as K-major A / B
      const uint64_t dv_a = smem_desc_sw128(sb + kKvOffV, 16, 1024);
      const uint64_t dk_mn = smem_desc_sw128(sb + kKvOffK, 8192, 1024);  // K as MN-major B (dQ)
      // S^T and dP^T of sub-step s into buffer s & 1
      auto issue_scores = [&](int s) -> bool {
        const int i = s >> 1, hf = s & 1;
        const uint32_t st = i & 1;
        if (hf == 0 && !mbar_wait_warp(bar(kKvBarFull + st), (i >> 1) & 1)) return false;
        if (s >= 2 && !mbar_wait_warp(bar(kKvBarXFree + hf), ((s >> 1) - 1) & 1)) return false;
        tc_fence_after();
        const uint32_t qa = sb + kKvOffRing + st * kKvStage + hf * kHalfTile;
        const uint64_t dqh = smem_desc_sw128(qa, 16, 1024);
        const uint64_t ddoh = smem_desc_sw128(qa + kTile, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk)
          umma_bf16_ss_elect(tmem + kColS + hf * 64, dk_a + 2 * kk, dqh + 2 * kk, kIdS64, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk)
          umma_bf16_ss_elect(tmem + kColDP + hf * 64, dv_a + 2 * kk, ddoh + 2 * kk, kIdS64, kk > 0 ? 1u : 0u);
        tc_commit_elect(bar(kKvBarS + hf));
        return true;
      };
      if (ok && nsub > 0) ok = issue_scores(0);
      if (ok && nsub > 1) ok = issue_scores(1);
      for (int s = 0; ok && s < nsub; ++s) {
        const int i = s >> 1, hf = s & 1;
        const uint32_t st = i & 1;
        ok = mbar_wait_warp(bar(kKvBarP + hf), (s >> 1) & 1);
        if (!ok || __any_sync(0xffffffffu, *abort_f != 0)) break;
        tc_fence_after();
        // dV += P^T dO_h, dK += dS^T Q_h (A from TMEM, B = the half's 64 rows, MN-major)
        const uint32_t qa = sb + kKvOffRing + st * kKvStage + hf * kHalfTile;
        const uint64_t bq = smem_desc_sw128(qa, 8192, 1024);
        const uint64_t bdo = smem_desc_sw128(qa + kTile, 8192, 1024);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_ts_elect(tmem + kColDV, tmem + kColS + hf * 64 + kk * 8, bdo + 128 * kk, kIdAcc,
                             (s > 0 || kk > 0) ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 4; ++kk)
          umma_bf16_ts_elect(tmem + kColDK, tmem + kColDP + hf * 64 + kk * 8, bq + 128 * kk, kIdAcc,
                             (s > 0 || kk > 0) ? 1u : 0u);
        tc_commit_elect(bar(kKvBarXFree + hf));
        if (hf == 1) {
          // dQ_i = dS K: A = dS (query-major, two 64-key halves), B = K MN-major
          if (i > 0) ok = mbar_wait_warp(bar(kKvBarDqFree), (i - 1) & 1);
          if (!ok) break;
          tc_fence_after();
          const uint32_t ds = sb + kKvOffDS + (i & 1) * 2 * kTile;
#pragma unroll
          for (int kk = 0; kk < kBT / 16; ++kk) {
            const uint64_t da = smem_desc_sw128(ds + (kk >> 2) * kTile, 16, 1024) + 2 * (kk & 3);
            umma_bf16_ss_elect(tmem + kColDQ, da, dk_mn + 128 * kk, kIdAcc, kk > 0 ? 1u : 0u);
          }
          tc_commit_elect(bar(kKvBarDqFull));
          tc_commit_elect(bar(kKvBarEmpty + st));  // the tile's Q and dO are read
        }
        if (s + 2 < nsub) {
          ok = issue_scores(s + 2);
          if (!ok) break;
        }
      }
      if (!ok && lane == 0) {
        *abort_f = 1;
        bwd_error(p.status);
      }
      tc_commit_elect(bar(kKvBarFin));
    }
  } else if (warp < 12) {
    setmaxnreg_inc<200>();
    // ---------------------------------------------------------- compute
    // The tables are built here, while the first tiles load and the first
    // products run (only these warpgroups read them).
    {
      const int ct = static_cast<int>(threadIdx.x) - 128;  // 0 .. 255
      if constexpr (MODE == 0) {
        load_bucket_bias(bsm, p, h, ct);
        named_bar_sync(3, 256);
        build_bias_copies(tab, bsm, p, true, ct, 256, 3, bk);
        for (int x = ct; x < tab_len(R); x += 256) hist[x] = 0.f;
        for (int x = ct; x < kMaxT5Buckets; x += 256) hist_b[x] = 0.f;
      }
      if (ct < 16) red[ct] = 0.f;
      named_bar_sync(3, 256);
    }
    const int hf = (warp - 4) >> 2;  // query half 0 / 1 of every tile = TMEM buffer
    const int t = ((warp & 3) << 5) | lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int key = j0 + t;
    const bool key_ok = key < p.Lk;
    float alibi = 0.f;
    if constexpr (MODE == 3) alibi = __ldg(p.slopes + h) * kLog2e;
    float sumL = 0.f, sumR = 0.f, dsl = 0.f;  // T5 saturated sides; ALiBi slope gradient
    float kfl = 0.f, kfr = 0.f;               // DeBERTa: dS over the queries beyond the band
    const float2 sc2 = make_float2(p.scale_log2, p.scale_log2);
    bool err = false;
    for (int s = hf, c = 0; s < nsub; s += 2, ++c) {
      const int i = s >> 1;
      const int q0 = (first + i) * kBT + hf * 64;  // first query of the sub-step
      bool ok = mbar_wait(bar(kKvBarS + hf), c & 1);
      err = __any_sync(0xffffffffu, !ok);
      // leave together: the TMEM loads and stores below are warp-collective
      if (err || __any_sync(0xffffffffu, *abort_f != 0)) break;
      tc_fence_after();
      // this sub-step's lse and D, staged with the query tile
      const float* lse_s = reinterpret_cast<const float*>(smem + kKvOffRing + (i & 1) * kKvStage + 2 * kTile) + hf * 64;
      const float* dd_s = lse_s + 128;
      uint32_t sr[64], dr[64];
      tmem_ld32(tmem + lane_base + kColS + hf * 64, *reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld32(tmem + lane_base + kColS + hf * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld32(tmem + lane_base + kColDP + hf * 64, *reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
      tmem_ld32(tmem + lane_base + kColDP + hf * 64 + 32, *reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&sr[0]));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&sr[32]));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&dr[0]));
      tmem_ld_wait(*reinterpret_cast<uint32_t(*)[32]>(&dr[32]));
      // offsets key - query position: rb - c for column c, rel_lo .. rel_hi
      // over the sub-step (uniform classes)
      const int rb = key - q0 - p.q_offset;
      const int rel_hi = j0 + kBT - 1 - (q0 + p.q_offset), rel_lo = j0 - (q0 + 63 + p.q_offset);
      const bool nomask = j0 + kBT <= p.Lk && q0 + 64 <= p.Lq && (!p.causal || rel_hi <= 0);
      const bool far_l = (MODE == 0 && rel_hi <= -R) || ((MODE == 1 || MODE == 2) && rel_hi <= -p.kc);
      const bool far_r = (MODE == 0 && p.t5.bidir && rel_lo >= R) || ((MODE == 1 || MODE == 2) && rel_lo >= p.kc);
      // dS goes to shared memory as it is formed: the dQ product of tile
      // i - 2 must have read this buffer
      if (i >= 2) {
        ok = mbar_wait(bar(kKvBarDsFree + (i & 1)), ((i >> 1) - 1) & 1);
        err = __any_sync(0xffffffffu, !ok);
        if (err) break;
      }
      // Every 16 columns: P^T and dS^T (bf16 pairs) over the first half of
      // the buffer's S^T and dP^T columns, and dS into the query-major tile
      // (row q = query, key t in half t / 64, K-major, 128-byte swizzle).
      const uint32_t ds_base = sb + kKvOffDS + (i & 1) * 2 * kTile + (t >> 6) * kTile +
                               static_cast<uint32_t>(t & 7) * 2u + static_cast<uint32_t>(hf) * 64u * 128u;
      const uint32_t kc = static_cast<uint32_t>((t & 63) >> 3);
      auto emit = [&](int g, const uint32_t (&pp)[8], const uint32_t (&pd)[8]) {
        tmem_st8(tmem + lane_base + kColS + hf * 64 + 8 * g, pp);
        tmem_st8(tmem + lane_base + kColDP + hf * 64 + 8 * g, pd);
#pragma unroll
        for (int e = 0; e < 8; ++e) {
#pragma unroll
          for (int u = 0; u < 2; ++u) {
            const uint32_t q = static_cast<uint32_t>(16 * g + 2 * e + u);  // row within the half
            st_shared_u16(ds_base + q * 128u + ((kc ^ (q & 7u)) << 4),
                          static_cast<uint16_t>(u ? (pd[e] >> 16) : (pd[e] & 0xffffu)));
          }
        }
      };
      // T5 near or masked sub-steps: dS summed per offset along the warp's
      // diagonals, d = l - c for lane l and column c (offset: its key - q0
      // - q_offset - c = d + the offset of lane 0 at column 0). The dS
      // values are kept in dr[] as they are formed; then four independent
      // chains (columns 16k .. 16k + 15) run their diagonal sums side by
      // side: after each column a chain's sums shift one lane up, the one
      // leaving lane 31 (d = 32 - c: no lane of this chain meets it again)
      // parked in the warp's strip at entry d + 63, and after its last
      // column the 32 sums still in its lanes (d = l - 16k - 15) are added
      // to their entries. The 95 entries d = -63 .. 31 then go into the
      // histogram with three shared atomics per lane. Histogram indices past
      // the table (offsets beyond the saturation distance on a masked tile)
      // clamp to its ends, which lie in the same saturated buckets.
      const int hbase = (key - lane) - q0 - p.q_offset + R + kTabPad;
      const int hlast = tab_len(R) - 1;
      float* wstrip = strip + (warp - 4) * 96;
      auto diag_sums = [&]() {
        for (int e = lane; e < 96; e += 32) wstrip[e] = 0.f;
        __syncwarp();
        float a[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int i = 0; i < 16; ++i) {
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            const int c = 16 * k + i;
            if (i > 0) {
              if (lane == 31) wstrip[95 - c] = a[k];
              a[k] = __shfl_up_sync(0xffffffffu, a[k], 1);
              if (lane == 0) a[k] = 0.f;
            }
            a[k] += __uint_as_float(dr[c]);
          }
        }
#pragma unroll
        for (int k = 3; k >= 0; --k) {
          __syncwarp();
          wstrip[lane + 48 - 16 * k] += a[k];
        }
        __syncwarp();
        for (int e = lane; e < 95; e += 32) atomicAdd(&hist[min(max(hbase + e - 63, 0), hlast)], wstrip[e]);
        __syncwarp();  // read before the next sub-step writes
      };
      bool diag = false;  // a T5 sub-step that summed per offset
      if (nomask && (MODE != 3 ? (far_l || far_r) : (rel_hi <= 0 || rel_lo >= 0))) {
        // one bias per row (T5 beyond the saturation distance), or ALiBi with
        // every key on one side: the logit is s * scale + g (c - rb) with
        // g = -slope (keys behind: |rel| = c - rb) or +slope (ahead: rb - c)
        // F index of offset o: R + kTabPad - o. Shaw beyond the clip: each
        // column's query takes its T and U of the side's end offset.
        // DeBERTa beyond the band: the key's saturated p2c value is the
        // constant, the column's c2p value joins lse (lse - c2p)
        float bc = 0.f;
        if constexpr (MODE == 0) bc = far_l ? tab[2 * R + kTabPad] : tab[kTabPad];
        if constexpr (MODE == 2)
          bc = __ldg(p.p2c_ends + (static_cast<size_t>(bh) * 2 + (far_l ? 0 : 1)) * p.ends_pitch + min(key, p.Lk - 1));
        // Shaw: lse - T and D - U of the side's end offset stand for lse and D
        const float* lse_f = (MODE == 1 || MODE == 2) ? tab + (i & 1) * 512 + (far_l ? 0 : 128) + hf * 64 : lse_s;
        const float* dd_f = (MODE == 1 || MODE == 2) ? lse_f + 256 : dd_s;
        const float g = MODE == 0 ? 0.f : (rel_hi <= 0 ? -alibi : alibi);
        const float2 g2 = make_float2(g, g);
        const float nrb = -static_cast<float>(rb);
        float2 acc = make_float2(0.f, 0.f);  // T5: dS of the side; ALiBi: sum dS (c - rb)
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
          uint32_t pp[8], pd[8];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const int q = 4 * gi + qq;
            const float4 L = *reinterpret_cast<const float4*>(lse_f + 4 * q);
            const float4 D = *reinterpret_cast<const float4*>(dd_f + 4 * q);
            float2 off0 = make_float2(bc - L.x, bc - L.y), off1 = make_float2(bc - L.z, bc - L.w);
            float2 cm0 = make_float2(0.f, 0.f), cm1 = make_float2(0.f, 0.f);
            if constexpr (MODE == 3) {
              cm0 = __fadd2_rn(make_float2(static_cast<float>(4 * q), static_cast<float>(4 * q + 1)),
                               make_float2(nrb, nrb));
              cm1 = __fadd2_rn(make_float2(static_cast<float>(4 * q + 2), static_cast<float>(4 * q + 3)),
                               make_float2(nrb, nrb));
              off0 = __ffma2_rn(cm0, g2, off0);
              off1 = __ffma2_rn(cm1, g2, off1);
            }
            float2 e0 = __ffma2_rn(make_float2(__uint_as_float(sr[4 * q]), __uint_as_float(sr[4 * q + 1])), sc2, off0);
            float2 e1 =
                __ffma2_rn(make_float2(__uint_as_float(sr[4 * q + 2]), __uint_as_float(sr[4 * q + 3])), sc2, off1);
            e0.x = ex2_approx(e0.x);
            e0.y = ex2_approx(e0.y);
            e1.x = ex2_approx(e1.x);
            e1.y = ex2_approx(e1.y);
            const float2 t0 = __fadd2_rn(make_float2(__uint_as_float(dr[4 * q]), __uint_as_float(dr[4 * q + 1])),
                                         make_float2(-D.x, -D.y));
            const float2 t1 = __fadd2_rn(
                make_float2(__uint_as_float(dr[4 * q + 2]), __uint_as_float(dr[4 * q + 3])), make_float2(-D.z, -D.w));
            const float2 d0 = __fmul2_rn(e0, t0), d1 = __fmul2_rn(e1, t1);
            if constexpr (MODE == 0 || MODE == 2) {
              acc = __fadd2_rn(acc, __fadd2_rn(d0, d1));
            } else if constexpr (MODE == 3) {
              acc = __ffma2_rn(d0, cm0, acc);
              acc = __ffma2_rn(d1, cm1, acc);
            }
            pp[2 * qq] = pack_bf16x2(e0.x, e0.y);
            pp[2 * qq + 1] = pack_bf16x2(e1.x, e1.y);
            pd[2 * qq] = pack_bf16x2(d0.x, d0.y);
            pd[2 * qq + 1] = pack_bf16x2(d1.x, d1.y);
          }
          emit(gi, pp, pd);
        }
        const float a = acc.x + acc.y;
        if constexpr (MODE == 0) {
          if (far_l)
            sumL += a;
          else
            sumR += a;
        } else if constexpr (MODE == 2) {
          if (far_l)
            kfl += a;
          else
            kfr += a;
        } else if constexpr (MODE == 3) {
          dsl += rel_hi <= 0 ? a : -a;  // |rel| = c - rb behind, rb - c ahead
        }
      } else if (MODE == 0 && nomask) {
        diag = true;
        // T5 inside the saturation distance, no mask: the biases of the
        // columns' offsets rb - c read 4 at a time from F (index R + kTabPad
        // - rb + c), every dS added to its offset's sum (consecutive keys:
        // consecutive entries, no two lanes on one)
        const float4* bw = tab_window(tab, R, R + kTabPad - rb);
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
          uint32_t pp[8], pd[8];
#pragma unroll
          for (int qq = 0; qq < 4; ++qq) {
            const int q = 4 * gi + qq;
            const float4 L = *reinterpret_cast<const float4*>(lse_s + 4 * q);
            const float4 D = *reinterpret_cast<const float4*>(dd_s + 4 * q);
            const float4 b4 = bw[q];
            float2 e0 = __ffma2_rn(make_float2(__uint_as_float(sr[4 * q]), __uint_as_float(sr[4 * q + 1])), sc2,
                                   make_float2(b4.x - L.x, b4.y - L.y));
            float2 e1 = __ffma2_rn(make_float2(__uint_as_float(sr[4 * q + 2]), __uint_as_float(sr[4 * q + 3])), sc2,
                                   make_float2(b4.z - L.z, b4.w - L.w));
            e0.x = ex2_approx(e0.x);
            e0.y = ex2_approx(e0.y);
            e1.x = ex2_approx(e1.x);
            e1.y = ex2_approx(e1.y);
            const float2 t0 = __fadd2_rn(make_float2(__uint_as_float(dr[4 * q]), __uint_as_float(dr[4 * q + 1])),
                                         make_float2(-D.x, -D.y));
            const float2 t1 = __fadd2_rn(
                make_float2(__uint_as_float(dr[4 * q + 2]), __uint_as_float(dr[4 * q + 3])), make_float2(-D.z, -D.w));
            const float2 d0 = __fmul2_rn(e0, t0), d1 = __fmul2_rn(e1, t1);
            dr[4 * q] = __float_as_uint(d0.x);  // dS, for the per-offset sums
            dr[4 * q + 1] = __float_as_uint(d0.y);
            dr[4 * q + 2] = __float_as_uint(d1.x);
            dr[4 * q + 3] = __float_as_uint(d1.y);
            pp[2 * qq] = pack_bf16x2(e0.x, e0.y);
            pp[2 * qq + 1] = pack_bf16x2(e1.x, e1.y);
            pd[2 * qq] = pack_bf16x2(d0.x, d0.y);
            pd[2 * qq + 1] = pack_bf16x2(d1.x, d1.y);
          }
          emit(gi, pp, pd);
        }
      } else {
        diag = MODE == 0;
        // per element: masks, the bias of each offset, T5 dS summed per
        // offset; Shaw reads each column's T and U rows (the statistics
        // kernel's, through L2)
        const size_t srow = (static_cast<size_t>(bh) * p.lq_pad + q0) * p.nr;
#pragma unroll
        for (int gi = 0; gi < 4; ++gi) {
          uint32_t pp[8], pd[8];
#pragma unroll
          for (int e = 0; e < 16; e += 2) {
            float pv[2], dsv[2];
#pragma unroll
            for (int u = 0; u < 2; ++u) {
              const int cc = 16 * gi + e + u;
              const int rel = rb - cc;
              // branch-free: masked elements take 2^-inf = 0 (a divergent
              // branch around each exponential costs several times the work)
              const bool valid = key_ok & (q0 + cc < p.Lq) & (!p.causal | (rel <= 0));
              float b, ua = 0.f;
              if constexpr (MODE == 0) {
                b = tab[min(max(R + kTabPad - rel, 0), tab_len(R) - 1)];
              } else if constexpr (MODE == 1) {
                const size_t o = srow + static_cast<size_t>(cc) * p.nr + (min(max(rel, -p.kc), p.kc) + p.kc);
                b = __ldg(p.shT + o);
                ua = __ldg(p.shU + o);
              } else if constexpr (MODE == 2) {
                b = deberta_bias(p, bh, q0 + cc, q0 + cc + p.q_offset, key, rel + p.kc);
              } else {
                b = -alibi * fabsf(static_cast<float>(rel));
              }
              const float s2 = fmaf(__uint_as_float(sr[cc]), p.scale_log2, b - lse_s[cc]);
              const float pr = ex2_approx(valid ? s2 : -INFINITY);
              const float ds = pr * (__uint_as_float(dr[cc]) + ua - dd_s[cc]);
              pv[u] = pr;
              dsv[u] = ds;
              if constexpr (MODE == 0) {
                dr[cc] = __float_as_uint(ds);  // for the per-offset sums
              } else if constexpr (MODE == 2) {
                // inside the band each (query, table row) and (key, table
                // row) meets one score: c2p row 2k - m, p2c row m
                const int m = rel + p.kc, k2 = 2 * p.kc;
                if (m >= 1 && m < k2) {
                  const __nv_bfloat16 v = __float2bfloat16_rn(ds);
                  p.dSQ[(static_cast<size_t>(bh) * p.lq_pad + q0 + cc) * k2 + (k2 - m)] = v;
                  p.dSK[(static_cast<size_t>(bh) * p.lk_pad + key) * k2 + m] = v;
                  // the saturated rows' band members also in fp32: the fold
                  // adds the far sums to them before rounding (the sums can
                  // nearly cancel them)
                  if (m == 1) p.rowm1[static_cast<size_t>(bh) * p.lq_pad + q0 + cc] = ds;
                  if (m == k2 - 1) p.keymk[static_cast<size_t>(bh) * p.lk_pad + key] = ds;
                }
                kfl += m <= 0 ? ds : 0.f;
                kfr += m >= k2 ? ds : 0.f;
              } else if constexpr (MODE == 3) {
                dsl = fmaf(ds, fabsf(static_cast<float>(rel)), dsl);
              }
            }
            pp[e / 2] = pack_bf16x2(pv[0], pv[1]);
            pd[e / 2] = pack_bf16x2(dsv[0], dsv[1]);
          }
          emit(gi, pp, pd);
        }
      }
      if (MODE == 0 && diag) diag_sums();
      tmem_st_wait();
      tc_fence_before();
      fence_async_smem();
      mbar_arrive(bar(kKvBarP + hf));
    }
    if (err) {
      *abort_f = 1;
      bwd_error(p.status);
    }
    // ---- the bias gradient of this CTA
    named_bar_sync(3, 256);  // every histogram add of both warpgroups is done
    if constexpr (MODE == 0) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        sumL += __shfl_xor_sync(0xffffffffu, sumL, o);
        sumR += __shfl_xor_sync(0xffffffffu, sumR, o);
      }
      if (lane == 0) {
        atomicAdd(&red[0], sumL);
        atomicAdd(&red[1], sumR);
      }
      const int ct = tid - 128;  // 0 .. 255
      // per-offset sums into their buckets: 32 consecutive offsets per warp
      // and round, summed per run of one bucket (a segmented scan over the
      // lanes), one shared atomic per run; a bucket covers a run of offsets
      // on each side, so few atomics meet on one address
      for (int x0 = ct - lane; x0 < tab_len(R); x0 += 256) {
        const int xo = x0 + lane;
        const bool in = xo < tab_len(R);
        float v = in ? hist[xo] : 0.f;
        const int b = in ? static_cast<int>(bk[xo]) : -1;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const float vo = __shfl_up_sync(0xffffffffu, v, o);
          const int bo = __shfl_up_sync(0xffffffffu, b, o);
          if (lane >= o && bo == b) v += vo;
        }
        const int bn = __shfl_down_sync(0xffffffffu, b, 1);
        if (b >= 0 && (lane == 31 || bn != b) && v != 0.f) atomicAdd(&hist_b[b], v);
      }
      named_bar_sync(3, 256);
      if (ct == 0) {
        atomicAdd(&hist_b[t5_bucket_dev(-R, p.t5)], red[0]);
        atomicAdd(&hist_b[t5_bucket_dev(R, p.t5)], red[1]);
      }
      named_bar_sync(3, 256);
      if (!*abort_f)
        for (int xb = ct; xb < p.nb; xb += 256)
          if (hist_b[xb] != 0.f) atomicAdd(p.dbias + xb * p.H + h, hist_b[xb]);
    } else if constexpr (MODE == 3) {
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) dsl += __shfl_xor_sync(0xffffffffu, dsl, o);
      if (lane == 0) atomicAdd(&red[2], dsl);
      named_bar_sync(3, 256);
      if (tid == 128 && !*abort_f && red[2] != 0.f) atomicAdd(p.dslopes + h, -red[2]);
    }
    if constexpr (MODE == 2) {  // this query half's far sums of the key
      const size_t kf = (static_cast<size_t>(hf) * gridDim.y + bh) * 2 * p.lk_pad + key;
      p.keyfar[kf] = kfl;
      p.keyfar[kf + p.lk_pad] = kfr;
    }
    // ---- dV (warpgroup 0) and dK (warpgroup 1; DeBERTa: fp32, the table
    // term is added later)
    // warp-uniform: the TMEM loads below are warp-collective
    const bool fin = __all_sync(0xffffffffu, mbar_wait(bar(kKvBarFin), 0) && *abort_f == 0);
    tc_fence_after();
    const bool f32k = MODE == 2 && hf == 1;
    __nv_bfloat16* dst = (hf == 0 ? p.dV : p.dK) + (static_cast<size_t>(bh) * p.Lk + key) * kHeadDim;
    uint4* d4 = reinterpret_cast<uint4*>(dst);
    float4* f4 = reinterpret_cast<float4*>(p.dKacc + (static_cast<size_t>(bh) * p.Lk + key) * kHeadDim);
    if (nsub > 0 && fin) {
      uint32_t a[32], b[32];  // every lane loads (warp-collective); rows past Lk are not stored
      tmem_ld32(tmem + lane_base + (hf == 0 ? kColDV : kColDK), a);
      tmem_ld32(tmem + lane_base + (hf == 0 ? kColDV : kColDK) + 32, b);
      tmem_ld_wait(a);
      tmem_ld_wait(b);
      const float mul = hf == 0 ? 1.f : p.scale;
      if (key_ok && f32k) {
#pragma unroll
        for (int v = 0; v < 16; ++v) {
          const uint32_t* r = v < 8 ? &a[v * 4] : &b[(v - 8) * 4];
          f4[v] = make_float4(__uint_as_float(r[0]) * mul, __uint_as_float(r[1]) * mul,
                              __uint_as_float(r[2]) * mul, __uint_as_float(r[3]) * mul);
        }
      } else if (key_ok) {
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
    } else if (nsub == 0 && key_ok) {  // no query sees this key
      if (f32k) {
#pragma unroll
        for (int v = 0; v < 16; ++v) f4[v] = make_float4(0.f, 0.f, 0.f, 0.f);
      } else {
#pragma unroll
        for (int v = 0; v < 8; ++v) d4[v] = make_uint4(0u, 0u, 0u, 0u);
      }
    }
    if (!fin && lane == 0) bwd_error(p.status);
  } else {
    setmaxnreg_dec<56>();
    // ---------------------------------------------------------- dQ accumulation
    // Each dQ_i (fp32, scaled) goes through the tile's dS buffer, which its
    // dQ product has finished reading, as two 128 x 32 boxes (128-byte
    // swizzle, conflict-free row writes), and one thread adds them into the
    // fp32 accumulator with bulk tensor reductions; once those have read the
    // buffer, it is released to the compute warpgroups (DsFree).
    const int t = ((warp & 3) << 5) | lane;
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    bool pending = false;  // thread 0 of the warpgroup has bulk reductions in flight
    for (int i = 0; i < ntiles; ++i) {
      const bool ok = mbar_wait(bar(kKvBarDqFull), i & 1);
      if (__any_sync(0xffffffffu, !ok || *abort_f != 0)) {  // the whole warp leaves
        if (!ok) bwd_error(p.status);
        *abort_f = 1;
        break;
      }
      tc_fence_after();
      const uint32_t buf = sb + kKvOffDS + (i & 1) * 2 * kTile;
#pragma unroll
      for (int half = 0; half < 2; ++half) {  // columns 32 half .. 32 half + 31: box `half`
        uint32_t a[32];
        tmem_ld32(tmem + lane_base + kColDQ + 32 * half, a);
        tmem_ld_wait(a);
        if (half == 1) {
          tc_fence_before();
          mbar_arrive(bar(kKvBarDqFree));  // the issuer may write the next dQ tile
        }
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          const uint32_t off = static_cast<uint32_t>(half) * kTile + static_cast<uint32_t>(t) * 128u +
                               ((static_cast<uint32_t>(ch) ^ (t & 7u)) << 4);
          const float sc = p.scale;
          asm volatile("st.shared.v4.f32 [%0], {%1, %2, %3, %4};" ::"r"(buf + off),
                       "f"(__uint_as_float(a[4 * ch]) * sc), "f"(__uint_as_float(a[4 * ch + 1]) * sc),
                       "f"(__uint_as_float(a[4 * ch + 2]) * sc), "f"(__uint_as_float(a[4 * ch + 3]) * sc)
                       : "memory");
        }
      }
      fence_async_smem();
      mbar_arrive(bar(kKvBarDqStage));
      if (t == 0) {
        bool staged = mbar_wait(bar(kKvBarDqStage), i & 1);
        if (staged) {
          const int q0 = (first + i) * kBT;
          tma_reduce_add_3d(&tmAcc, buf, 0, q0, bh);
          tma_reduce_add_3d(&tmAcc, buf + kTile, 32, q0, bh);
          bulk_commit();
          pending = true;
          bulk_wait_read();
        } else {
          *abort_f = 1;
          bwd_error(p.status);
        }
        mbar_arrive(bar(kKvBarDsFree + (i & 1)));
      }
    }
    if (t == 0 && pending) bulk_wait_all();  // no bulk operation outlives the CTA
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ================================================================ dQ to bf16
__global__ void relpos_bwd_dq_convert_kernel(const float4* __restrict__ acc, uint2* __restrict__ dq, size_t n4) {
  griddep_wait();
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 v = acc[i];
    dq[i] = make_uint2(pack_bf16x2(v.x, v.y), pack_bf16x2(v.z, v.w));
  }
}

// T5: four bias-table copies; Shaw: a_K and a_V, the rows' T and U and the
// two warpgroups' per-offset sums (nr floats per row each); then the merge
// buffer and the T5 bias per bucket
// ================================================================ Shaw: dQ and the tables' gradients
// One CTA per 128-row query tile and head. dQ_i = the accumulated (scaled)
// dS K part + scale * sum_r BdS_i[r] a_K[r], to bf16; and the tile's partial
// sums over its rows of BdS_i[r] q_i (da_K) and BP_i[r] dO_i (da_V).
constexpr int kShThreads = 256;
constexpr int kShQs = 68;  // row stride of the staged Q and dO rows (floats; 16-byte aligned rows)

__global__ void __launch_bounds__(kShThreads) relpos_bwd_shaw_final_kernel(const BwdParams p) {
  extern __shared__ float4 shf4[];
  float* shf = reinterpret_cast<float*>(shf4);
  const int nrel = 2 * p.kc + 1, nr = p.nr;
  float* qf = shf;                // [128][kShQs]
  float* of = qf + kBT * kShQs;   // [128][kShQs]
  float* aKf = of + kBT * kShQs;  // [2k + 1][64]
  float* bds = aKf + nrel * 64;   // [128][nr]
  float* bps = bds + kBT * nr;    // [128][nr]
  const int tid = threadIdx.x;
  const int tile = blockIdx.x, bh = blockIdx.y, i0 = tile * kBT;
  const int rows = min(kBT, p.Lq - i0);
  griddep_wait();
  for (int e = tid; e < nrel * 64; e += kShThreads) aKf[e] = __bfloat162float(p.aK[e]);
  const size_t g0 = (static_cast<size_t>(bh) * p.lq_pad + i0) * nr;
  for (int e = tid; e < kBT * nr; e += kShThreads) {
    bds[e] = p.shBdS[g0 + e];
    bps[e] = p.shBP[g0 + e];
  }
  for (int e = tid; e < kBT * 8; e += kShThreads) {  // 8 runs of 8 values per row
    const int r = e >> 3, ch = e & 7;
    uint4 uq = make_uint4(0u, 0u, 0u, 0u), uo = uq;
    if (r < rows) {
      const size_t off = (static_cast<size_t>(bh) * p.Lq + i0 + r) * kHeadDim + ch * 8;
      uq = *reinterpret_cast<const uint4*>(p.Qp + off);
      uo = *reinterpret_cast<const uint4*>(p.dOp + off);
    }
    const uint32_t wq[4] = {uq.x, uq.y, uq.z, uq.w}, wo[4] = {uo.x, uo.y, uo.z, uo.w};
    float fq[8], fo[8];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wq[k]));
      const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wo[k]));
      fq[2 * k] = a.x;
      fq[2 * k + 1] = a.y;
      fo[2 * k] = b.x;
      fo[2 * k + 1] = b.y;
    }
    float4* dq4 = reinterpret_cast<float4*>(qf + r * kShQs + ch * 8);
    float4* do4 = reinterpret_cast<float4*>(of + r * kShQs + ch * 8);
    dq4[0] = make_float4(fq[0], fq[1], fq[2], fq[3]);
    dq4[1] = make_float4(fq[4], fq[5], fq[6], fq[7]);
    do4[0] = make_float4(fo[0], fo[1], fo[2], fo[3]);
    do4[1] = make_float4(fo[4], fo[5], fo[6], fo[7]);
  }
  __syncthreads();
  {  // dQ: a row per thread pair, columns 4 u + 8 v (u = the thread's half)
    const int r = tid >> 1, u = tid & 1;
    if (r < rows) {
      const size_t off = (static_cast<size_t>(bh) * p.Lq + i0 + r) * kHeadDim + 4 * u;
      float4 acc[8];
#pragma unroll
      for (int v = 0; v < 8; ++v) acc[v] = *reinterpret_cast<const float4*>(p.dQacc + off + 8 * v);
#pragma unroll 1
      for (int k = 0; k < nrel; ++k) {
        const float w = bds[r * nr + k] * p.scale;
        const float4* a4 = reinterpret_cast<const float4*>(aKf + k * 64 + 4 * u);
#pragma unroll
        for (int v = 0; v < 8; ++v) {
          const float4 a = a4[2 * v];
          acc[v] = make_float4(fmaf(w, a.x, acc[v].x), fmaf(w, a.y, acc[v].y), fmaf(w, a.z, acc[v].z),
                               fmaf(w, a.w, acc[v].w));
        }
      }
#pragma unroll
      for (int v = 0; v < 8; ++v)
        *reinterpret_cast<uint2*>(p.dQ + off + 8 * v) =
            make_uint2(pack_bf16x2(acc[v].x, acc[v].y), pack_bf16x2(acc[v].z, acc[v].w));
    }
  }
  {  // the tile's partial table gradients: columns 4 c4 .. 4 c4 + 3 and the
     // offsets kg, kg + 16, kg + 32 per thread
    const int c4 = tid & 15, kg = tid >> 4;
    float4 sk[3], sv[3];
#pragma unroll
    for (int m = 0; m < 3; ++m) sk[m] = sv[m] = make_float4(0.f, 0.f, 0.f, 0.f);
    int kk[3];
#pragma unroll
    for (int m = 0; m < 3; ++m) kk[m] = min(kg + 16 * m, nrel - 1);  // clamped: read, not written
#pragma unroll 2
    for (int r = 0; r < rows; ++r) {
      const float4 q = *reinterpret_cast<const float4*>(qf + r * kShQs + 4 * c4);
      const float4 o = *reinterpret_cast<const float4*>(of + r * kShQs + 4 * c4);
#pragma unroll
      for (int m = 0; m < 3; ++m) {
        const float a = bds[r * nr + kk[m]], b = bps[r * nr + kk[m]];
        sk[m] = make_float4(fmaf(a, q.x, sk[m].x), fmaf(a, q.y, sk[m].y), fmaf(a, q.z, sk[m].z), fmaf(a, q.w, sk[m].w));
        sv[m] = make_float4(fmaf(b, o.x, sv[m].x), fmaf(b, o.y, sv[m].y), fmaf(b, o.z, sv[m].z), fmaf(b, o.w, sv[m].w));
      }
    }
    float* part = p.shPart + (static_cast<size_t>(bh) * gridDim.x + tile) * 2 * nrel * 64;
#pragma unroll
    for (int m = 0; m < 3; ++m) {
      const int k = kg + 16 * m;
      if (k < nrel) {
        *reinterpret_cast<float4*>(part + k * 64 + 4 * c4) = sk[m];
        *reinterpret_cast<float4*>(part + (nrel + k) * 64 + 4 * c4) = sv[m];
      }
    }
  }
}

// da_K (scaled) and da_V: one table row per CTA, summed over every tile's
// partial in a fixed order (deterministic)
__global__ void __launch_bounds__(kShThreads) relpos_bwd_shaw_reduce_kernel(const BwdParams p, int nparts) {
  __shared__ float red[kShThreads];
  const int nrel = 2 * p.kc + 1;
  const int row = blockIdx.x;  // 0 .. 2 nrel - 1: da_K rows, then da_V rows
  const int tid = threadIdx.x, c = tid & 63, g = tid >> 6;
  griddep_wait();
  const size_t stride = static_cast<size_t>(2) * nrel * 64;
  const float* src = p.shPart + static_cast<size_t>(row) * 64 + c;
  float s[8];
#pragma unroll
  for (int u = 0; u < 8; ++u) s[u] = 0.f;
  int q = g;
  for (; q + 28 < nparts; q += 32) {
#pragma unroll
    for (int u = 0; u < 8; ++u) s[u] += src[static_cast<size_t>(q + 4 * u) * stride];
  }
  for (int u = 0; q < nparts; q += 4, ++u) s[u & 7] += src[static_cast<size_t>(q) * stride];
  red[tid] = ((s[0] + s[1]) + (s[2] + s[3])) + ((s[4] + s[5]) + (s[6] + s[7]));
  __syncthreads();
  if (g == 0) {
    const float v = (red[c] + red[64 + c]) + (red[128 + c] + red[192 + c]);
    if (row < nrel)
      p.daK[row * 64 + c] = v * p.scale;
    else
      p.daV[(row - nrel) * 64 + c] = v;
  }
}

// DeBERTa: the rows' and keys' dS beyond the band into the saturated table
// rows of the gathered dS (c2p row 2k - 1 takes the keys far behind, row 0
// those far ahead; p2c row 0 the queries with m <= 0, row 2k - 1 those with
// m >= 2k), after the dK / dV kernel has scattered the band; a saturated row
// that also holds a band member (c2p 2k - 1: m = 1; p2c 2k - 1: m = 2k - 1)
// sums it in fp32 first
__global__ void __launch_bounds__(256) relpos_bwd_deberta_fold_kernel(const BwdParams p) {
  griddep_wait();
  const int k2 = 2 * p.kc;
  const size_t nbh = static_cast<size_t>(p.B) * p.H;
  const size_t nq = nbh * p.lq_pad, nk = nbh * p.lk_pad;
  for (size_t x = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; x < nq + nk;
       x += static_cast<size_t>(gridDim.x) * blockDim.x) {
    if (x < nq) {
      const size_t bh = x / p.lq_pad, i = x % p.lq_pad;
      const float L = p.rowfar[bh * 2 * p.lq_pad + i], R = p.rowfar[(bh * 2 + 1) * p.lq_pad + i];
      __nv_bfloat16* row = p.dSQ + x * k2;
      row[k2 - 1] = __float2bfloat16_rn(p.rowm1[x] + L);
      row[0] = __float2bfloat16_rn(R);
    } else {
      const size_t y = x - nq, bh = y / p.lk_pad, j = y % p.lk_pad;
      const size_t a0 = bh * 2 * p.lk_pad + j, a1 = (nbh + bh) * 2 * p.lk_pad + j;  // query halves 0, 1
      const float KL = p.keyfar[a0] + p.keyfar[a1];
      const float KR = p.keyfar[a0 + p.lk_pad] + p.keyfar[a1 + p.lk_pad];
      __nv_bfloat16* row = p.dSK + y * k2;
      row[0] = __float2bfloat16_rn(KL);
      row[k2 - 1] = __float2bfloat16_rn(p.keymk[y] + KR);
    }
  }
}

uint32_t shaw_final_smem_bytes(int nr) {
  const uint32_t nrel = static_cast<uint32_t>(nr) - 1u;
  return (2u * kBT * kShQs + nrel * 64u + 2u * kBT * static_cast<uint32_t>(nr)) * 4u;
}

uint32_t stats_smem_bytes(int mode, int R, int nr) {
  const uint32_t tab = mode == 0 ? 4u * static_cast<uint32_t>(tab_stride(R)) * 4u : 0u;
  const uint32_t shaw = mode == 1 ? (64u * 64u + 6u * 128u * static_cast<uint32_t>(nr)) * 4u : 0u;
  const uint32_t aux = mode == 1 ? StLayout<1>::kOffAux : StLayout<0>::kOffAux;
  return 1024u + aux + tab + shaw + (7u * 128u + kMaxT5Buckets) * 4u;
}

// T5: four bias-table copies, the per-offset sums, the compute warps'
// strips and the bucket of each offset (ALiBi: none); bucket sums, 16 floats
// of side / slope partials and the biases per bucket
// (Shaw: the two ring stages' end values)
uint32_t dkdv_smem_bytes(int mode, int R) {
  const uint32_t t5 =
      mode == 0 ? (4u * static_cast<uint32_t>(tab_stride(R)) + static_cast<uint32_t>(tab_len(R)) + 8u * 96u) * 4u +
                      ((static_cast<uint32_t>(tab_len(R)) + 15u) & ~15u)
                : (mode == 1 || mode == 2) ? 2u * 2048u : 0u;
  return 1024u + kKvOffAux + t5 + (2u * kMaxT5Buckets + 16u) * 4u;
}

template <typename K>
cudaError_t launch_pdl(K kern, dim3 grid, dim3 block, uint32_t smem, cudaStream_t stream, const CUtensorMap& a,
                       const CUtensorMap& b, const CUtensorMap& c, const CUtensorMap& d, const BwdParams& p) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, a, b, c, d, p);
}

// the fp32 accumulator [rows, 64] to bf16
cudaError_t launch_convert(const float* acc, __nv_bfloat16* out, size_t rows, cudaStream_t stream) {
  const size_t n4 = rows * kHeadDim / 4;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  size_t blocks = (n4 + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  cfg.gridDim = dim3(static_cast<unsigned>(blocks > 0 ? blocks : 1));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, relpos_bwd_dq_convert_kernel, reinterpret_cast<const float4*>(acc),
                            reinterpret_cast<uint2*>(out), n4);
}

cublasHandle_t cublas_handle_locked(int dev) {
  static cublasHandle_t handles[64] = {};
  if (dev < 0 || dev >= 64) return nullptr;
  if (!handles[dev] && cublasCreate(&handles[dev]) != CUBLAS_STATUS_SUCCESS) handles[dev] = nullptr;
  return handles[dev];
}

// DeBERTa after the dK / dV kernel: the far sums folded into the gathered dS,
// then four plain GEMMs per batch element (batched over the heads; cuBLAS,
// bf16 operands, fp32 accumulation) add the table terms to dQ and dK and form
// the tables' gradients, then dQ and dK go to bf16. With s the logit scale:
//   dQ_bh += s dSQ_bh Pk_h,   dK_bh += s dSK_bh Pq_h,
//   dPk_h += s dSQ_bh^T Q_bh, dPq_h += s dSK_bh^T K_bh   (summed over b)
// (row-major operands; cuBLAS sees their transposes).
cudaError_t launch_deberta_tail(const BwdParams& p, cudaStream_t stream) {
  {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(152 * 4);
    cfg.blockDim = dim3(256);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    const cudaError_t e = cudaLaunchKernelEx(&cfg, relpos_bwd_deberta_fold_kernel, p);
    if (e != cudaSuccess) return e;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  static std::mutex mu;
  {
    std::lock_guard<std::mutex> lock(mu);
    cublasHandle_t h = cublas_handle_locked(dev);
    if (!h || cublasSetStream(h, stream) != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
    const int k2 = 2 * p.kc, H = p.H;
    const float s = p.scale, one = 1.f;
    const long long sq = static_cast<long long>(p.lq_pad) * k2, sk = static_cast<long long>(p.lk_pad) * k2;
    for (int b = 0; b < p.B; ++b) {
      const size_t bh0 = static_cast<size_t>(b) * H;
      const __nv_bfloat16* dsq = p.dSQ + bh0 * sq;
      const __nv_bfloat16* dsk = p.dSK + bh0 * sk;
      cublasStatus_t st = cublasGemmStridedBatchedEx(
          h, CUBLAS_OP_N, CUBLAS_OP_N, kHeadDim, p.Lq, k2, &s, p.Pk, CUDA_R_16BF, H * kHeadDim, kHeadDim, dsq,
          CUDA_R_16BF, k2, sq, &one, p.dQacc + bh0 * p.Lq * kHeadDim, CUDA_R_32F, kHeadDim,
          static_cast<long long>(p.Lq) * kHeadDim, H, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
      if (st == CUBLAS_STATUS_SUCCESS)
        st = cublasGemmStridedBatchedEx(
            h, CUBLAS_OP_N, CUBLAS_OP_N, kHeadDim, p.Lk, k2, &s, p.Pq, CUDA_R_16BF, H * kHeadDim, kHeadDim, dsk,
            CUDA_R_16BF, k2, sk, &one, p.dKacc + bh0 * p.Lk * kHeadDim, CUDA_R_32F, kHeadDim,
            static_cast<long long>(p.Lk) * kHeadDim, H, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
      if (st == CUBLAS_STATUS_SUCCESS)
        st = cublasGemmStridedBatchedEx(
            h, CUBLAS_OP_N, CUBLAS_OP_T, kHeadDim, k2, p.Lq, &s, p.Qp + bh0 * p.Lq * kHeadDim, CUDA_R_16BF, kHeadDim,
            static_cast<long long>(p.Lq) * kHeadDim, dsq, CUDA_R_16BF, k2, sq, &one, p.dPk, CUDA_R_32F,
            H * kHeadDim, kHeadDim, H, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
      if (st == CUBLAS_STATUS_SUCCESS)
        st = cublasGemmStridedBatchedEx(
            h, CUBLAS_OP_N, CUBLAS_OP_T, kHeadDim, k2, p.Lk, &s, p.Kp + bh0 * p.Lk * kHeadDim, CUDA_R_16BF, kHeadDim,
            static_cast<long long>(p.Lk) * kHeadDim, dsk, CUDA_R_16BF, k2, sk, &one, p.dPq, CUDA_R_32F,
            H * kHeadDim, kHeadDim, H, CUBLAS_COMPUTE_32F, CUBLAS_GEMM_DEFAULT);
      if (st != CUBLAS_STATUS_SUCCESS) return cudaErrorUnknown;
    }
  }
  const size_t nbh = static_cast<size_t>(p.B) * p.H;
  cudaError_t e = launch_convert(p.dQacc, p.dQ, nbh * p.Lq, stream);
  if (e == cudaSuccess) e = launch_convert(p.dKacc, p.dK, nbh * p.Lk, stream);
  return e;
}

template <int MODE>
cudaError_t launch_bwd_mode(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                            const CUtensorMap& tmdO, const CUtensorMap& tmAcc, const BwdParams& p,
                            cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return cudaErrorInvalidDevice;
  static std::atomic<uint64_t> attr_set{0};
  const uint64_t bit = dev < 64 ? (uint64_t(1) << dev) : 0;
  if (!bit || !(attr_set.load() & bit)) {
    cudaError_t e = cudaFuncSetAttribute(relpos_bwd_stats_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(stats_smem_bytes(MODE, kMaxR, 2 * kMaxShawK + 2)));
    if (e == cudaSuccess)
      e = cudaFuncSetAttribute(relpos_bwd_dkdv_kernel<MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(dkdv_smem_bytes(MODE, kMaxR)));
    if (e == cudaSuccess && MODE == 1)
      e = cudaFuncSetAttribute(relpos_bwd_shaw_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(shaw_final_smem_bytes(2 * kMaxShawK + 2)));
    if (e != cudaSuccess) return e;
    attr_set.fetch_or(bit);
  }
  const unsigned BH = static_cast<unsigned>(p.B * p.H);
  cudaError_t e = launch_pdl(relpos_bwd_stats_kernel<MODE>, dim3((p.Lq + kBT - 1) / kBT, BH), dim3(kStThreads),
                             stats_smem_bytes(MODE, p.R, p.nr), stream, tmQ, tmK, tmV, tmdO, p);
  if (e != cudaSuccess) return e;
  {
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((p.Lk + kBT - 1) / kBT, BH);
    cfg.blockDim = dim3(kKvThreads);
    cfg.dynamicSmemBytes = dkdv_smem_bytes(MODE, p.R);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, relpos_bwd_dkdv_kernel<MODE>, tmQ, tmK, tmV, tmdO, tmAcc, p);
    if (e != cudaSuccess) return e;
  }
  if constexpr (MODE == 2) return launch_deberta_tail(p, stream);
  if constexpr (MODE == 1) {
    const int nqt = (p.Lq + kBT - 1) / kBT;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nqt), BH);
    cfg.blockDim = dim3(kShThreads);
    cfg.dynamicSmemBytes = shaw_final_smem_bytes(p.nr);
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, relpos_bwd_shaw_final_kernel, p);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(static_cast<unsigned>(2 * (2 * p.kc + 1)));
    cfg.dynamicSmemBytes = 0;
    return cudaLaunchKernelEx(&cfg, relpos_bwd_shaw_reduce_kernel, p, static_cast<int>(BH) * nqt);
  }
  const size_t n4 = static_cast<size_t>(BH) * p.Lq * kHeadDim / 4;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  size_t blocks = (n4 + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  cfg.gridDim = dim3(static_cast<unsigned>(blocks > 0 ? blocks : 1));
  cfg.blockDim = dim3(256);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, relpos_bwd_dq_convert_kernel, reinterpret_cast<const float4*>(p.dQacc),
                            reinterpret_cast<uint2*>(p.dQ), n4);
}

}  // namespace

int bwd_max_R() { return kMaxR; }
int bwd_max_shaw_k() { return kMaxShawK; }

cudaError_t launch_bwd(int mode, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const CUtensorMap& tmdO, const CUtensorMap& tmAcc, const BwdParams& p,
                       cudaStream_t stream) {
  if (mode == 0) {
    if (p.R < 1 || p.R > kMaxR || p.nb > kMaxT5Buckets) return cudaErrorInvalidValue;
    return launch_bwd_mode<0>(tmQ, tmK, tmV, tmdO, tmAcc, p, stream);
  }
  if (mode == 1) {
    if (p.kc < 1 || p.kc > kMaxShawK || p.nr != 2 * p.kc + 2) return cudaErrorInvalidValue;
    return launch_bwd_mode<1>(tmQ, tmK, tmV, tmdO, tmAcc, p, stream);
  }
  if (mode == 2) {
    if (p.kc < 1 || !p.band || !p.dSQ || !p.dSK) return cudaErrorInvalidValue;
    return launch_bwd_mode<2>(tmQ, tmK, tmV, tmdO, tmAcc, p, stream);
  }
  if (mode == 3) return launch_bwd_mode<3>(tmQ, tmK, tmV, tmdO, tmAcc, p, stream);
  return cudaErrorInvalidValue;
}

}  // namespace relpos
