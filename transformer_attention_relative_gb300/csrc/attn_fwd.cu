// attn_fwd.cu -- fused relative-position attention forward for sm_103a.
//
// One CTA owns a 128-row query tile of one (batch, head) and streams the
// key/value tiles of that head through shared memory:
//
//   warp 0      TMA producer: Q tile once, then K_j / V_j into a 3-stage ring.
//   warp 1      tcgen05 issuer (one thread): S_j = Q K_j^T into one of two
//               TMEM score buffers, then O += P_j V_j once the softmax has
//               produced P_j. Also allocates / frees the 512 TMEM columns.
//   warps 2-5   softmax warpgroup: thread t owns query row t (TMEM lane t).
//               It reads its S row from TMEM, adds the relative term (from a
//               shared-memory table, never a materialised L x L tensor),
//               masks, keeps the running max / sum, writes bf16 P to shared
//               memory for the next tensor-core product, and finally
//               normalises O and stores it.
//
// The relative term follows "Relative Position Embeddings, in depth": T5 adds
// a per-head scalar by bucket of the key-minus-query offset ("T5: one scalar
// per head, looked up by bucket"); Shaw adds q_i . a_K[clip(j - i)] to the
// logit and sum_j p_ij a_V[clip(j - i)] to the output ("Shaw et al.").
// Because both depend on the offset only, a tile whose offsets all lie beyond
// the saturation distance gets one constant (T5) or one per-row constant
// (Shaw) instead of per-element lookups.
//
// Softmax runs in the log2 domain with a lazily updated running maximum: the
// output accumulator in TMEM is rescaled only when a row's maximum grows by
// more than 2^8, which keeps every P value <= 256 and is exact because the
// final division uses the same stale maximum.

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"
#include "relpos_common.cuh"
#include "relpos_internal.h"

namespace relpos {
namespace {

constexpr int kBM = 128;         // query rows per CTA
constexpr int kBN = 128;         // keys per tile
constexpr int kStages = 3;       // K/V ring depth
constexpr int kThreads = 192;    // 6 warps
constexpr uint32_t kTileBytes = kBM * kHeadDim * 2;  // 16 KB: 128 rows x 128 B
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffK = kOffQ + kTileBytes;
constexpr uint32_t kOffV = kOffK + kStages * kTileBytes;
constexpr uint32_t kOffP = kOffV + kStages * kTileBytes;  // 128 x 128 bf16 = 32 KB
constexpr uint32_t kOffBar = kOffP + 2 * kTileBytes;
constexpr uint32_t kOffAux = kOffBar + 256;
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemS = 0;    // two score buffers: columns 0..127, 128..255
constexpr uint32_t kTmemO = 256;  // output accumulator: columns 256..319
constexpr float kRescaleThreshold = 8.0f;  // log2 units

// barrier slots (8 bytes each) inside the kOffBar block
enum : uint32_t {
  kBarQFull = 0,
  kBarKFull = 1,                   // + stage
  kBarVFull = kBarKFull + kStages,  // + stage
  kBarKVEmpty = kBarVFull + kStages,
  kBarSFull = kBarKVEmpty + kStages,  // + buffer (2)
  kBarPFull = kBarSFull + 2,
  kBarODone = kBarPFull + 1,
  kBarFinal = kBarODone + 1,
  kNumBars = kBarFinal + 1,
};
constexpr uint32_t kOffTmemSlot = kNumBars * 8;
constexpr uint32_t kOffAbort = kOffTmemSlot + 4;

constexpr uint32_t kIdescQK = idesc_bf16_f32(kBM, kBN, 0, 0);       // Q, K both K-major
constexpr uint32_t kIdescPV = idesc_bf16_f32(kBM, kHeadDim, 0, 1);  // P K-major, V MN-major

// byte offset of 16-byte chunk `c` of row `r` in a 128-byte-swizzled tile
// of 128-byte rows (the layout TMA writes and the tensor core reads)
RP_DEVI uint32_t sw128_offset(int r, int c) {
  return static_cast<uint32_t>((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}

RP_DEVI void record_error(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}

template <int MODE, bool OUT_F32>
__global__ void __launch_bounds__(kThreads, 1)
    relpos_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                      const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmO,
                      const FwdParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_addr);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qt = gridDim.x - 1 - blockIdx.x;  // longest (causal) tiles first
  const int bh = blockIdx.y;
  const int h = bh % p.H;
  const int i0 = qt * kBM;

  // number of key tiles this query tile visits
  int last_key = p.Lk - 1;
  if (p.causal) {
    const int last_row = min(i0 + kBM - 1, p.Lq - 1);
    last_key = min(last_key, last_row + p.q_offset);
  }
  const int n_kv = last_key / kBN + 1;

  auto bar = [&](uint32_t i) { return sbase + kOffBar + i * 8; };
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffBar + kOffAbort);

  if (threadIdx.x == 0) {
    for (uint32_t i = 0; i < kNumBars; ++i)
      mbar_init(bar(i), i == kBarPFull ? 128u : 1u);  // every softmax thread arrives on P
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(sbase + kOffBar + kOffTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffBar + kOffTmemSlot);

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tmQ);
      tma_prefetch_desc(&tmK);
      tma_prefetch_desc(&tmV);
      mbar_arrive_expect_tx(bar(kBarQFull), kTileBytes);
      tma_load_3d(sbase + kOffQ, &tmQ, bar(kBarQFull), 0, i0, bh);
      bool err = false;
      int issued = 0;
      for (int j = 0; j < n_kv; ++j) {
        const int st = j % kStages;
        if (j >= kStages) {
          if (!mbar_wait(bar(kBarKVEmpty + st), ((j / kStages) - 1) & 1)) {
            err = true;
            break;
          }
        }
        mbar_arrive_expect_tx(bar(kBarKFull + st), kTileBytes);
        tma_load_3d(sbase + kOffK + st * kTileBytes, &tmK, bar(kBarKFull + st), 0, j * kBN, bh);
        mbar_arrive_expect_tx(bar(kBarVFull + st), kTileBytes);
        tma_load_3d(sbase + kOffV + st * kTileBytes, &tmV, bar(kBarVFull + st), 0, j * kBN, bh);
        issued = j + 1;
      }
      if (err) {
        record_error(p.status, -4);
        *abort_flag = 1;
      }
      // never leave with copies in flight: wait (bounded) for the last loads
      for (int j = (issued > kStages ? issued - kStages : 0); j < issued; ++j) {
        const int st = j % kStages;
        mbar_wait(bar(kBarKFull + st), (j / kStages) & 1, 100000000ull);
        mbar_wait(bar(kBarVFull + st), (j / kStages) & 1, 100000000ull);
      }
      mbar_wait(bar(kBarQFull), 0, 100000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = mbar_wait(bar(kBarQFull), 0);
      tc_fence_after();
      const uint32_t q_addr = sbase + kOffQ;
      auto issue_qk = [&](int j) {
        const int st = j % kStages;
        const uint32_t k_addr = sbase + kOffK + st * kTileBytes;
        const uint32_t d = tmem + kTmemS + (j & 1) * kBN;
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk) {
          const uint64_t a = smem_desc_sw128(q_addr + kk * 32, 16, 1024);
          const uint64_t b = smem_desc_sw128(k_addr + kk * 32, 16, 1024);
          umma_bf16_ss(d, a, b, kIdescQK, kk > 0 ? 1u : 0u);
        }
        tc_commit(bar(kBarSFull + (j & 1)));
      };
      if (ok) ok = mbar_wait(bar(kBarKFull + 0), 0);
      tc_fence_after();
      if (ok) issue_qk(0);
      for (int j = 0; ok && j < n_kv; ++j) {
        if (j + 1 < n_kv) {
          const int st1 = (j + 1) % kStages;
          ok = mbar_wait(bar(kBarKFull + st1), ((j + 1) / kStages) & 1);
          tc_fence_after();
          if (!ok) break;
          issue_qk(j + 1);
        }
        ok = mbar_wait(bar(kBarPFull), j & 1);
        tc_fence_after();
        if (!ok) break;
        const int st = j % kStages;
        ok = mbar_wait(bar(kBarVFull + st), (j / kStages) & 1);
        tc_fence_after();
        if (!ok) break;
        const uint32_t v_addr = sbase + kOffV + st * kTileBytes;
        const uint32_t p_addr = sbase + kOffP;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint64_t a = smem_desc_sw128(p_addr + (kk >> 2) * kTileBytes + (kk & 3) * 32, 16, 1024);
          const uint64_t b = smem_desc_sw128(v_addr + kk * 2048, 8192, 1024);
          umma_bf16_ss(tmem + kTmemO, a, b, kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        }
        tc_commit(bar(kBarODone));
        tc_commit(bar(kBarKVEmpty + st));
      }
      if (!ok) {
        record_error(p.status, -4);
        *abort_flag = 1;
      }
      // all issued tensor-core work has finished before TMEM is released
      tc_commit(bar(kBarFinal));
      mbar_wait(bar(kBarFinal), 0, 100000000ull);
    }
  } else {
    // ------------------------------------------------------------ softmax
    const int t = ((warp & 3) << 5) | lane;  // row == TMEM lane
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const int prow = i0 + t + p.q_offset;    // absolute query position
    const int p_lo = i0 + p.q_offset;
    const float sl2 = p.scale_log2;
    bool err = false;

    float* tab = reinterpret_cast<float*>(smem + kOffAux);
    float add_left = 0.f, add_right = 0.f;
    int kc = 0;
    float* qa = nullptr;   // Shaw: this row's q . a_K[r] (log2 units)
    float* wbin = nullptr; // Shaw: this row's attention mass per clipped offset
    const __nv_bfloat16* aK_s = nullptr;
    const __nv_bfloat16* aV_s = nullptr;
    float mass_l = 0.f, mass_r = 0.f;

    if constexpr (MODE == 0) {
      // per-head bias by offset, offsets -t5_tab_off .. tab_len-1-t5_tab_off
      for (int x = t; x < p.t5_tab_len; x += 128) {
        const int b = t5_bucket_dev(x - p.t5_tab_off, p.t5);
        tab[x] = __ldg(p.bias + b * p.H + h) * kLog2e;
      }
      add_left = __ldg(p.bias + t5_bucket_dev(-p.t5_R, p.t5) * p.H + h) * kLog2e;
      add_right = __ldg(p.bias + t5_bucket_dev(p.t5_R, p.t5) * p.H + h) * kLog2e;
      named_bar_sync(1, 128);
    } else if constexpr (MODE == 1) {
      kc = p.kclip;
      const int nrel = 2 * kc + 1;
      const int tbl_bytes = nrel * kHeadDim * 2;
      uint8_t* aux = smem + kOffAux;
      aK_s = reinterpret_cast<const __nv_bfloat16*>(aux);
      aV_s = reinterpret_cast<const __nv_bfloat16*>(aux + ((tbl_bytes + 15) & ~15));
      float* qa_all = reinterpret_cast<float*>(aux + 2 * ((tbl_bytes + 15) & ~15));
      float* w_all = qa_all + 128 * nrel;
      {
        const uint4* srcK = reinterpret_cast<const uint4*>(p.aK);
        const uint4* srcV = reinterpret_cast<const uint4*>(p.aV);
        uint4* dK = reinterpret_cast<uint4*>(aux);
        uint4* dV = reinterpret_cast<uint4*>(aux + ((tbl_bytes + 15) & ~15));
        for (int x = t; x < tbl_bytes / 16; x += 128) {
          dK[x] = __ldg(srcK + x);
          dV[x] = __ldg(srcV + x);
        }
      }
      named_bar_sync(1, 128);
      qa = qa_all + t * nrel;
      wbin = w_all + t * nrel;
      if (!mbar_wait(bar(kBarQFull), 0)) err = true;
      err = __any_sync(0xffffffffu, err);
      if (!err) {
        float qf[kHeadDim];
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint32_t a, b, cc, d;
          ld_shared_v4(sbase + kOffQ + sw128_offset(t, c), a, b, cc, d);
          const uint32_t w4[4] = {a, b, cc, d};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const __nv_bfloat162 v2 = *reinterpret_cast<const __nv_bfloat162*>(&w4[e]);
            qf[c * 8 + 2 * e] = __bfloat162float(v2.x);
            qf[c * 8 + 2 * e + 1] = __bfloat162float(v2.y);
          }
        }
        for (int r = 0; r < nrel; ++r) {
          const __nv_bfloat162* row = reinterpret_cast<const __nv_bfloat162*>(aK_s + r * kHeadDim);
          float acc0 = 0.f, acc1 = 0.f;
#pragma unroll
          for (int e = 0; e < kHeadDim / 2; ++e) {
            const float2 f = __bfloat1622float2(row[e]);
            acc0 = fmaf(qf[2 * e], f.x, acc0);
            acc1 = fmaf(qf[2 * e + 1], f.y, acc1);
          }
          qa[r] = (acc0 + acc1) * sl2;
          wbin[r] = 0.f;
        }
      }
    }

    float m_run = -INFINITY;
    float l_run = 0.f;
    const float kNegInf = -INFINITY;

    for (int j = 0; j < n_kv && !err; ++j) {
      const int j0 = j * kBN;
      bool ok = mbar_wait(bar(kBarSFull + (j & 1)), (j >> 1) & 1);
      err = __any_sync(0xffffffffu, !ok);
      if (err) break;
      tc_fence_after();

      __syncwarp();
      uint32_t sr[4][32];
      const uint32_t s_addr = tmem + lane_base + kTmemS + (j & 1) * kBN;
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld32(s_addr + q * 32, sr[q]);
#pragma unroll
      for (int q = 0; q < 4; ++q) tmem_ld_wait(sr[q]);

      float x[128];
      // ---- logits in log2 units with the relative term
      if constexpr (MODE == 0) {
        const int rel_hi = j0 + kBN - 1 - p_lo;          // largest offset in the tile
        const int rel_lo = j0 - (p_lo + kBM - 1);        // smallest
        const bool far_l = rel_hi <= -p.t5_R;
        const bool far_r = p.t5.bidir && rel_lo >= p.t5_R;
        if (far_l || far_r) {
          const float a = far_l ? add_left : add_right;
#pragma unroll
          for (int c = 0; c < 128; ++c) x[c] = fmaf(__uint_as_float(sr[c >> 5][c & 31]), sl2, a);
        } else {
          const float* tp = tab + (j0 - prow + p.t5_tab_off);
#pragma unroll
          for (int c = 0; c < 128; ++c) x[c] = fmaf(__uint_as_float(sr[c >> 5][c & 31]), sl2, tp[c]);
        }
      } else if constexpr (MODE == 1) {
        const int rel_hi = j0 + kBN - 1 - p_lo;
        const int rel_lo = j0 - (p_lo + kBM - 1);
        if (rel_hi <= -kc || rel_lo >= kc) {
          const float a = rel_hi <= -kc ? qa[0] : qa[2 * kc];
#pragma unroll
          for (int c = 0; c < 128; ++c) x[c] = fmaf(__uint_as_float(sr[c >> 5][c & 31]), sl2, a);
        } else {
          const int r0 = j0 - prow;
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const int r = min(max(r0 + c, -kc), kc) + kc;
            x[c] = fmaf(__uint_as_float(sr[c >> 5][c & 31]), sl2, qa[r]);
          }
        }
      }

      // ---- masking (causal, ragged key tail)
      const bool need_mask = (p.causal && j0 + kBN - 1 > p_lo) || (j0 + kBN > p.Lk);
      if (need_mask) {
        int lim = p.Lk - 1 - j0;
        if (p.causal) lim = min(lim, prow - j0);
#pragma unroll
        for (int c = 0; c < 128; ++c) x[c] = (c > lim) ? kNegInf : x[c];
      }

      // ---- running max with lazy rescale
      float mx0 = kNegInf, mx1 = kNegInf, mx2 = kNegInf, mx3 = kNegInf;
#pragma unroll
      for (int c = 0; c < 128; c += 4) {
        mx0 = fmaxf(mx0, x[c]);
        mx1 = fmaxf(mx1, x[c + 1]);
        mx2 = fmaxf(mx2, x[c + 2]);
        mx3 = fmaxf(mx3, x[c + 3]);
      }
      const float mx = fmaxf(fmaxf(mx0, mx1), fmaxf(mx2, mx3));
      const float m_new = fmaxf(m_run, mx);
      const bool resc = m_new > m_run + kRescaleThreshold;
      float alpha = 1.f;
      if (resc) {
        alpha = ex2_approx(m_run - m_new);
        m_run = m_new;
      }
      const float m_use = (m_run == kNegInf) ? 0.f : m_run;

      float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
#pragma unroll
      for (int c = 0; c < 128; c += 4) {
        x[c] = ex2_approx(x[c] - m_use);
        x[c + 1] = ex2_approx(x[c + 1] - m_use);
        x[c + 2] = ex2_approx(x[c + 2] - m_use);
        x[c + 3] = ex2_approx(x[c + 3] - m_use);
        s0 += x[c];
        s1 += x[c + 1];
        s2 += x[c + 2];
        s3 += x[c + 3];
      }
      const float tile_sum = (s0 + s1) + (s2 + s3);
      l_run = l_run * alpha + tile_sum;

      if constexpr (MODE == 1) {
        // value-side mass per clipped offset
        if (resc && j > 0) {
          for (int r = 0; r < 2 * kc + 1; ++r) wbin[r] *= alpha;
          mass_l *= alpha;
          mass_r *= alpha;
        }
        const int rel_hi = j0 + kBN - 1 - p_lo;
        const int rel_lo = j0 - (p_lo + kBM - 1);
        if (rel_hi <= -kc) {
          mass_l += tile_sum;
        } else if (rel_lo >= kc) {
          mass_r += tile_sum;
        } else {
          const int r0 = j0 - prow;
#pragma unroll
          for (int c = 0; c < 128; ++c) {
            const int rel = r0 + c;
            if (rel <= -kc) {
              mass_l += x[c];
            } else if (rel >= kc) {
              mass_r += x[c];
            } else {
              wbin[rel + kc] += x[c];
            }
          }
        }
      }

      // ---- previous P.V must be done before P and O are touched
      if (j > 0) {
        ok = mbar_wait(bar(kBarODone), (j - 1) & 1);
        err = __any_sync(0xffffffffu, !ok);
        if (err) break;
        tc_fence_after();
        __syncwarp();
        if (__any_sync(0xffffffffu, resc)) {
          uint32_t o[2][32];
          const uint32_t o_addr = tmem + lane_base + kTmemO;
          tmem_ld32(o_addr, o[0]);
          tmem_ld32(o_addr + 32, o[1]);
          tmem_ld_wait(o[0]);
          tmem_ld_wait(o[1]);
#pragma unroll
          for (int q = 0; q < 2; ++q)
#pragma unroll
            for (int c = 0; c < 32; ++c) o[q][c] = __float_as_uint(__uint_as_float(o[q][c]) * alpha);
          tmem_st32(o_addr, o[0]);
          tmem_st32(o_addr + 32, o[1]);
          tmem_st_wait();
        }
      }

      // ---- bf16 P into the 128-byte-swizzled K-major operand tile
#pragma unroll
      for (int ch = 0; ch < 16; ++ch) {
        const uint32_t addr = sbase + kOffP + (ch >> 3) * kTileBytes + sw128_offset(t, ch & 7);
        st_shared_v4(addr, pack_bf16x2(x[ch * 8 + 0], x[ch * 8 + 1]),
                     pack_bf16x2(x[ch * 8 + 2], x[ch * 8 + 3]),
                     pack_bf16x2(x[ch * 8 + 4], x[ch * 8 + 5]),
                     pack_bf16x2(x[ch * 8 + 6], x[ch * 8 + 7]));
      }
      fence_async_smem();
      tc_fence_before();
      mbar_arrive(bar(kBarPFull));
    }

    // ------------------------------------------------------------ epilogue
    if (!err) {
      const bool ok = mbar_wait(bar(kBarODone), (n_kv - 1) & 1);
      err = __any_sync(0xffffffffu, !ok);
    }
    if (err) {
      record_error(p.status, -4);
      *abort_flag = 1;
    }
    float o[kHeadDim];
    if (!err) {
      tc_fence_after();
      __syncwarp();
      uint32_t orr[2][32];
      const uint32_t o_addr = tmem + lane_base + kTmemO;
      tmem_ld32(o_addr, orr[0]);
      tmem_ld32(o_addr + 32, orr[1]);
      tmem_ld_wait(orr[0]);
      tmem_ld_wait(orr[1]);
#pragma unroll
      for (int c = 0; c < kHeadDim; ++c) o[c] = __uint_as_float(orr[c >> 5][c & 31]);
      if constexpr (MODE == 1) {
        wbin[0] += mass_l;
        wbin[2 * kc] += mass_r;
        for (int r = 0; r < 2 * kc + 1; ++r) {
          const float w = wbin[r];
          const __nv_bfloat162* row = reinterpret_cast<const __nv_bfloat162*>(aV_s + r * kHeadDim);
#pragma unroll
          for (int e = 0; e < kHeadDim / 2; ++e) {
            const float2 f = __bfloat1622float2(row[e]);
            o[2 * e] = fmaf(w, f.x, o[2 * e]);
            o[2 * e + 1] = fmaf(w, f.y, o[2 * e + 1]);
          }
        }
      }
      const float inv_l = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
      for (int c = 0; c < kHeadDim; ++c) o[c] *= inv_l;
    } else {
#pragma unroll
      for (int c = 0; c < kHeadDim; ++c) o[c] = 0.f;
    }
    if constexpr (OUT_F32) {
      const int row = i0 + t;
      if (!err && row < p.Lq) {
        float4* dst = reinterpret_cast<float4*>(static_cast<float*>(p.out) +
                                                (static_cast<size_t>(bh) * p.Lq + row) * kHeadDim);
#pragma unroll
        for (int c = 0; c < kHeadDim / 4; ++c)
          dst[c] = make_float4(o[4 * c], o[4 * c + 1], o[4 * c + 2], o[4 * c + 3]);
      }
    } else {
      // stage the bf16 tile in the (now idle) Q buffer, then one TMA store
#pragma unroll
      for (int c = 0; c < 8; ++c) {
        st_shared_v4(sbase + kOffQ + sw128_offset(t, c), pack_bf16x2(o[8 * c], o[8 * c + 1]),
                     pack_bf16x2(o[8 * c + 2], o[8 * c + 3]), pack_bf16x2(o[8 * c + 4], o[8 * c + 5]),
                     pack_bf16x2(o[8 * c + 6], o[8 * c + 7]));
      }
      fence_async_smem();
      named_bar_sync(1, 128);
      if (t == 0 && *abort_flag == 0) {
        tma_store_3d(&tmO, sbase + kOffQ, 0, i0, bh);
        tma_store_commit();
        tma_store_wait_read_all();
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

uint32_t fwd_smem_bytes(int mode, const FwdParams& p) {
  uint32_t aux = 0;
  if (mode == 0) {
    aux = static_cast<uint32_t>(p.t5_tab_len) * 4u;
  } else if (mode == 1) {
    const uint32_t nrel = 2u * p.kclip + 1u;
    const uint32_t tbl = (nrel * kHeadDim * 2u + 15u) & ~15u;
    aux = 2u * tbl + 2u * 128u * nrel * 4u;
  }
  return 1024u + kOffAux + ((aux + 15u) & ~15u);
}

cudaError_t launch_fwd(int mode, bool out_f32, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const CUtensorMap& tmO, const FwdParams& p,
                       cudaStream_t stream) {
  const uint32_t smem = fwd_smem_bytes(mode, p);
  dim3 grid((p.Lq + kBM - 1) / kBM, p.B * p.H);
  dim3 block(kThreads);
  void (*kern)(const CUtensorMap, const CUtensorMap, const CUtensorMap, const CUtensorMap,
               const FwdParams) = nullptr;
  if (mode == 0) {
    kern = out_f32 ? relpos_fwd_kernel<0, true> : relpos_fwd_kernel<0, false>;
  } else if (mode == 1) {
    kern = out_f32 ? relpos_fwd_kernel<1, true> : relpos_fwd_kernel<1, false>;
  } else {
    return cudaErrorNotSupported;
  }
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  kern<<<grid, block, smem, stream>>>(tmQ, tmK, tmV, tmO, p);
  return cudaGetLastError();
}

uint32_t fwd_max_smem_bytes() { return 232448u; }

}  // namespace relpos
