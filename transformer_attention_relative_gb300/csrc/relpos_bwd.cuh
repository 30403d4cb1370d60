// relpos_bwd.cuh -- parameter block, launcher and tcgen05 helper of the T5
// attention backward (attn_bwd.cu), kept apart from the headers the forward
// and decode kernels compile.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstdint>

#include "ptx.cuh"
#include "relpos_common.cuh"

namespace relpos {

constexpr int kMaxT5Buckets = 128;

// Backward of the T5-bias and the ALiBi attention (attn_bwd.cu)
struct BwdParams {
  int B, H, Lq, Lk;
  int causal, q_offset;
  float scale;       // 1 / sqrt(d)
  float scale_log2;  // scale times log2(e)
  // T5
  const float* bias;  // [nb, H]
  int nb;
  int R;  // |offset| >= R: the side's last bucket; offsets in (-R, R) get a table entry each (ALiBi: 0)
  T5Index t5;
  float* dbias;  // [nb, H], zeroed before the kernels, accumulated by the dK / dV kernel
  // ALiBi
  const float* slopes;  // [H]
  float* dslopes;       // [H], zeroed before the kernels
  // Shaw (mode 1): per query row, with rows padded to lq_pad and nr floats
  // per row (the 2k + 1 clipped offsets r, one spare)
  const __nv_bfloat16* aK;  // [2k + 1, 64]
  const __nv_bfloat16* aV;  // [2k + 1, 64]
  int kc, nr;               // clip k, nr = 2k + 2
  float* shT;               // [B*H, lq_pad, nr] q_i . a_K[r] * scale_log2 (statistics kernel)
  float* shU;               // [B*H, lq_pad, nr] dO_i . a_V[r]
  float* shEnds;            // [B*H, 4, lq_pad] lse - T[0], lse - T[2k], D - U[0], D - U[2k] of every row
                            // (DeBERTa: lse - the two saturated c2p values, D, D)
  float* shBP;              // [B*H, lq_pad, nr] sum of P_ij over the keys at clipped offset r
  float* shBdS;             // [B*H, lq_pad, nr] sum of dS_ij over them
  float* shPart;            // [query tiles * B*H, 2, 2k + 1, 64] per-tile partial da_K, da_V
  float* daK;               // [2k + 1, 64] fp32, written
  float* daV;               // [2k + 1, 64] fp32, written
  const __nv_bfloat16* Qp;   // [B*H, Lq, 64] (Shaw: the final kernel's rows)
  const __nv_bfloat16* dOp;  // [B*H, Lq, 64]
  // DeBERTa (mode 2; kc = k): the forward's band pre-pass arrays (c2p + p2c
  // inside the band, log2 units, bf16; the saturated c2p values per query row
  // and p2c values per key, fp32), and dS gathered by table row
  const __nv_bfloat16* band;  // [B*H, Lq, band_pitch], row i's offset m = j - p_i + k at ((p_i - k) & 7) + m
  int band_pitch;
  const float* c2p_const;     // [B*H, 2, const_pitch]: keys far behind (m <= 0), far ahead (m >= 2k)
  int const_pitch;
  const float* p2c_ends;      // [B*H, 2, ends_pitch]: the same two sides per key
  int ends_pitch;
  __nv_bfloat16* dSQ;         // [B*H, lq_pad, 2k]: sum of dS_ij over the keys with c2p row delta(i, j) = r (zeroed)
  __nv_bfloat16* dSK;         // [B*H, lk_pad, 2k]: sum over the queries with p2c row delta(j, i) = r (zeroed)
  int lk_pad;                 // Lk rounded up to a multiple of 128
  float* rowfar;              // [B*H, 2, lq_pad] per row: sum of dS over the keys with m <= 0, with m >= 2k
  float* keyfar;              // [2 query halves, B*H, 2, lk_pad] per key: the same over the queries
  float* rowm1;               // [B*H, lq_pad] dS of the row's key at m = 1, fp32 (zeroed)
  float* keymk;               // [B*H, lk_pad] dS of the key's query at m = 2k - 1, fp32 (zeroed)
  float* dKacc;               // [B*H, Lk, 64] fp32 dK (scaled), before the table terms
  const __nv_bfloat16* Kp;    // [B*H, Lk, 64]
  const __nv_bfloat16* Pk;    // [2k, H, 64]
  const __nv_bfloat16* Pq;    // [2k, H, 64]
  float* dPk;                 // [2k, H, 64] fp32, zeroed before the kernels
  float* dPq;                 // [2k, H, 64] fp32, zeroed before the kernels
  float* lse;    // [B*H, lq_pad] row log-sum-exp of the log2-scaled logits (stats kernel)
  float* Dr;     // [B*H, lq_pad] D_i = sum_j P_ij dP_ij (stats kernel)
  int lq_pad;    // Lq rounded up to a multiple of 128 (whole query tiles)
  float* dQacc;  // [B*H, Lq, 64] fp32, zeroed before the kernels: dQ summed over key tiles
  __nv_bfloat16* dQ;  // [B*H, Lq, 64]
  __nv_bfloat16* dK;  // [B*H, Lk, 64]
  __nv_bfloat16* dV;  // [B*H, Lk, 64]
  int* status;
};

// mode 0 (T5), 1 (Shaw), 2 (DeBERTa) or 3 (ALiBi): the row-statistics kernel
// (Shaw: also the per-row tables and the per-offset sums; DeBERTa: the rows'
// dS beyond the band), the dK / dV kernel (which also accumulates dQ and the
// T5 / ALiBi table gradient; DeBERTa: scatters dS by table row) and the dQ
// conversion (Shaw: with the a_K term, then the table gradients; DeBERTa:
// the table products, then dQ and dK); bwd_max_R is the largest T5
// saturation distance R they support, bwd_max_shaw_k the largest Shaw clip
int bwd_max_shaw_k();
int bwd_max_R();
// tmAcc: the fp32 dQ accumulator [B*H, Lq, 64] as 128-row x 32-column boxes
// (128-byte swizzle), the target of the dQ tiles' bulk reductions
cudaError_t launch_bwd(int mode, const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmV,
                       const CUtensorMap& tmdO, const CUtensorMap& tmAcc, const BwdParams& p,
                       cudaStream_t stream);

// 16 consecutive 32-bit TMEM columns of this thread's lane.
RP_DEVI void tmem_st16(uint32_t taddr, const uint32_t (&r)[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
      "r"(r[15])
      : "memory");
}

}  // namespace relpos
