// relpos_common.cuh -- parameter blocks shared by the host launchers and the
// kernels, and the device index generator (offset -> T5 bucket, Shaw clipped
// row, DeBERTa delta) that every kernel and the index test hook call.
#pragma once

#include <cuda_bf16.h>
#include <cstdint>

namespace relpos {

constexpr int kHeadDim = 64;
constexpr int kMaxT5Thresholds = 64;
constexpr float kLog2e = 1.4426950408889634f;

// T5 bucket generator ("Relative Position Embeddings, in depth", section
// "T5: one scalar per head, looked up by bucket"; "T5 Relative-Position
// Bias"). The host derives, once per call, the smallest distance at which
// each logarithmic bucket begins (thr[]), by evaluating the pages' double-
// precision log formula; the device then needs integer compares only, so
// its ids equal the formula's exactly.
struct T5Index {
  int bidir;   // 1: bidirectional (upper half for keys after the query)
  int slots;   // slots per direction: num_buckets / 2 (bidir) or num_buckets
  int exact;   // slots / 2 distances with a bucket each
  int nthr;    // slots - exact - 1 thresholds
  int thr[kMaxT5Thresholds];  // thr[q]: first distance with bucket >= exact + q + 1
};

__host__ __device__ inline int t5_bucket_dev(int rel, const T5Index& ix) {
  int base = 0, n;
  if (ix.bidir) {
    base = rel > 0 ? ix.slots : 0;
    n = rel < 0 ? -rel : rel;
  } else {
    n = rel < 0 ? -rel : 0;
  }
  if (n < ix.exact) return base + n;
  // the number of thresholds at or below n (they ascend): binary search
  int lo = 0, hi = ix.nthr;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (n >= ix.thr[mid]) {
      lo = mid + 1;
    } else {
      hi = mid;
    }
  }
  return base + ix.exact + lo;
}

// Shaw ("Relative Position Embeddings, in depth", section "Shaw et al."):
// offset key - query clipped to [-k, k], shifted to a row in [0, 2k].
__host__ __device__ inline int shaw_index_dev(int rel, int k) {
  int c = rel < -k ? -k : (rel > k ? k : rel);
  return c + k;
}

// DeBERTa ("DeBERTa > Relative Position Encoding", section "The Relative
// Position Formula"): r = i - j clipped to [-k, k - 1], shifted by k.
__host__ __device__ inline int deberta_delta_dev(int r, int k) {
  int c = r < -k ? -k : (r > k - 1 ? k - 1 : r);
  return c + k;
}

struct FwdParams {
  int B, H, Lq, Lk;
  int dh;  // head dimension: 64, or 128 (T5 and ALiBi)
  int causal, q_offset;
  float scale_log2;  // softmax scale times log2(e)
  void* out;
  int out_v8;  // out is 32-byte aligned: rows are written with 32-byte stores
  int stagger;  // offset the two softmax warpgroups by about half a tile
  int* status;
  const int* lengths;  // [B] valid rows and keys per batch element (right-padded batch), or null
  const int* key_pos;  // T5: [B*H, Lk] position of every key (explicit positions), or null
  // ALiBi
  const float* slopes;  // [H]
  // T5
  const float* bias;  // [num_buckets, H]
  int t5_R;           // |offset| >= R: the side's last bucket (no ordering left)
  int t5_tab_len;     // entries of the per-head bias-by-offset table
  int t5_tab_off;     // table index of offset 0
  int t5_tab_len4;    // t5_tab_len rounded up to a multiple of 4
  int t5_nb;          // num_buckets (<= 128)
  int t5_compact;     // one table copy read per entry (the four do not fit)
  T5Index t5;
  int npairs;         // 256-row query-tile pairs per head
  int nsplit;         // trailing pair items run as two split items each
  const __nv_bfloat16* Qg;  // Q in global memory (bf16 [B,H,Lq,dh])
  // Shaw
  const __nv_bfloat16* aK;  // [2k+1, 64]
  const __nv_bfloat16* aV;  // [2k+1, 64]
  // DeBERTa
  const __nv_bfloat16* Pk;  // [2k, H, 64]
  const __nv_bfloat16* Pq;  // [2k, H, 64]
  // DeBERTa (log2-scaled): band[bh][i][sh(i) + m] = c2p + p2c for key
  // j = i + m - k with 1 <= m <= 2k - 1, sh(i) = (i + q_offset - k) mod 8;
  // beyond the band c2p_const (C2P[i][2k - 1], C2P[i][0]) and p2c_ends
  // (P2C[j][0], P2C[j][2k - 1]) apply
  const __nv_bfloat16* band;  // [B*H, Lq, band_pitch]
  int band_pitch;             // 2k + 8 rounded up to a multiple of 8
  const float* c2p_const;     // [B*H, 2, const_pitch]
  int const_pitch;            // Lq rounded up to a multiple of 128
  const float* p2c_ends;      // [B*H, 2, ends_pitch]
  int ends_pitch;             // Lk rounded up to a multiple of 128
  int kclip;                 // Shaw / DeBERTa clip k
  int row_stride;            // Shaw: floats per row of the per-row tables (2k + 1 or 2k + 2)
};

// DeBERTa band pre-pass (deberta_band.cu)
struct BandParams {
  int BH, H, k, Lq, Lk, q_offset;
  float scale;                // applied to every product (softmax scale times log2 e)
  const __nv_bfloat16* K;     // [BH, Lk, 64]
  const __nv_bfloat16* Pq;    // [2k, H, 64]
  __nv_bfloat16* band;        // [BH, Lq, band_pitch]
  int band_pitch;
  float* c2p_const;           // [BH, 2, const_pitch]
  int const_pitch;
  float* ends;                // [BH, 2, ends_pitch]
  int ends_pitch;
  int* status;
};

// Transformer-XL operand pre-pass (txl_prep.cu)
struct TxlParams {
  int BH, H, Lq, Lk, q_offset;
  const __nv_bfloat16* Q;  // [BH, Lq, 64]
  const float* W;          // [H, 64, 64]: r(t) = W R(t), output index first
  const float* uv;         // [2, H, 64]: u, then v
  __nv_bfloat16* Q2;       // [BH, Lq, 128]: q + u, then a = W^T (q + v) rotated by w p
  __nv_bfloat16* Ksin;     // [Lk, 64]: (cos w_m j, sin w_m j)
  float omega[kHeadDim / 2];  // w_m = 10000^(-2m/64)
  int* status;               // device status word (bounded-wait failures)
};

struct DecodeParams {
  const __nv_bfloat16* Q;
  const __nv_bfloat16* K;
  const __nv_bfloat16* V;
  const float* bias;
  int B, H, Lq, Lk;
  int causal, q_offset;
  float scale_log2;
  int chunk;     // keys per partial
  int nchunks;
  float* part_o;   // [B*H*Lq, nchunks, 64]
  float* part_ml;  // [B*H*Lq, nchunks, 2]
  void* out;
  int out_f32;
  int t5_R;  // |offset| >= R: the side's last bucket; -1: ALiBi, bias holds the slopes [H]
  T5Index t5;
  const int* key_pos;  // [B*H, Lk] explicit key positions, or null (key j at position j)
};

}  // namespace relpos
