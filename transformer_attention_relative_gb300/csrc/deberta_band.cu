// deberta_band.cu -- the relative terms of DeBERTa attention, laid out by
// query row and key offset ("Relative Position Embeddings, in depth", section
// "DeBERTa: disentangled content and position"; the table index is delta of
// "DeBERTa > Relative Position Encoding", "The Relative Position Formula").
//
// For query position i and key j let m = j - i + k. Inside the band
// (1 <= m <= 2k - 1) neither table index is clipped:
//   c2p(i, j) = s * q_i . Pk[delta(i, j)],  delta(i, j) = 2k - m
//   p2c(i, j) = s * k_j . Pq[delta(j, i)],  delta(j, i) = m
// and this kernel writes their sum, rounded once to bf16, as
//   band[bh][i][sh(i) + m],  sh(i) = (i - k) mod 8 (i the absolute position),
// so that the attention kernel, which needs m = j0 - i + k ... + 127 for a
// 128-key tile starting at j0 (a multiple of 128), reads every row's window
// from a 16-byte aligned address. s is the softmax scale times log2(e).
// Outside the band both terms saturate: c2p is C2P[i][2k - 1] (keys far
// behind) or C2P[i][0] (far ahead), one value per row, written to c2p_const;
// p2c is P2C[j][0] or P2C[j][2k - 1], one value per key, written to ends.
//
// Grid z = 0: one CTA (128 threads, two per SM) per 128 query rows of one
// head, looping over chunks of 64 band columns. Per chunk, tcgen05.mma
// (M128 N64 K16) computes D1 = Q Pk^T over the chunk's 64 table rows (C2P,
// columns in reverse m order) and D2 = K Pq^T over the 256 keys from which
// the chunk's diagonal is taken. Row t, column u of the output takes
// D1[t][63 - u] + D2[t + u][u]: the P2C diagonal goes through a padded
// shared-memory slice (conflict-free for both the row-wise fill and the
// diagonal read), the row then through a shifted row buffer with an odd
// word pitch (conflict-free for the 32 rows a warp writes at once), from
// which whole 16-byte pieces are stored, eight lanes per row.
// Grid z = 1: the two P2C end columns of every key, on CUDA cores.

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"
#include "relpos_common.cuh"
#include "relpos_internal.h"

namespace relpos {
namespace {

constexpr int kRows = 128;  // query rows per CTA
constexpr int kChunk = 64;  // band columns per MMA group
constexpr uint32_t kTile = 128 * kHeadDim * 2;  // 16 KB: 128 rows x 128 B
constexpr uint32_t kHalf = kTile / 2;           // 64 rows
constexpr uint32_t kOffQ = 0;
constexpr uint32_t kOffPk = kOffQ + kTile;  // 64 Pk rows
constexpr uint32_t kOffPq = kOffPk + kHalf;  // 64 Pq rows
constexpr uint32_t kOffK = kOffPq + kHalf;   // 256 key rows
constexpr uint32_t kOpBytes = 2 * kHalf + 2 * kTile;
constexpr int kSlice = 32;  // band columns per diagonal slice
constexpr int kStageRows = kRows + kSlice - 1;
constexpr int kStagePitch = kSlice + 1;  // floats
constexpr uint32_t kOffStage = kOffK + 2 * kTile;
constexpr uint32_t kStageBytes = (kStageRows * kStagePitch * 4 + 1023) & ~1023u;
// row buffer pitch in words: with 43 the packed writes of a warp's 32 rows
// (shifted by (t + c) mod 8 columns) and the piece reads of four rows at a
// time both hit 32 distinct banks
constexpr int kOutWords = 43;
static_assert(2 * kOutWords >= kChunk + 8, "row buffer holds a chunk and its overhang");
constexpr uint32_t kOffOut = kOffStage + kStageBytes;
constexpr uint32_t kOutBytes = (kRows * kOutWords * 4 + 1023) & ~1023u;
constexpr uint32_t kOffBar = kOffOut + kOutBytes;
constexpr uint32_t kSmem = 1024 + kOffBar + 64;
static_assert(2 * kSmem <= 227 * 1024, "two CTAs per SM");
constexpr uint32_t kIdesc = idesc_bf16_f32(128, kChunk, 0, 0);
constexpr uint32_t kTmemCols = 256;  // D1 at 0, D2 (keys 0..127) at 64, (128..255) at 128
enum : uint32_t { kBarQ = 0, kBarOp = 1, kBarMma = 2, kNBar = 3 };
constexpr uint32_t kOffSlot = kNBar * 8;

// z = 1: P2C[j][0] and P2C[j][2k - 1] for the keys of this block
RP_DEVI void p2c_ends(const BandParams& bp, int bh) {
  const int j = blockIdx.x * kRows + threadIdx.x;
  if (j >= bp.Lk) return;
  const int h = bh % bp.H;
  const uint4* kr = reinterpret_cast<const uint4*>(bp.K + (static_cast<size_t>(bh) * bp.Lk + j) * kHeadDim);
  const __nv_bfloat162* p0 = reinterpret_cast<const __nv_bfloat162*>(bp.Pq + static_cast<size_t>(h) * kHeadDim);
  const __nv_bfloat162* p1 = reinterpret_cast<const __nv_bfloat162*>(
      bp.Pq + (static_cast<size_t>(2 * bp.k - 1) * bp.H + h) * kHeadDim);
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int c = 0; c < kHeadDim / 8; ++c) {
    const uint4 u = __ldg(kr + c);
    const uint32_t w4[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 kv = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
      const float2 a = __bfloat1622float2(p0[c * 4 + e]);
      const float2 b = __bfloat1622float2(p1[c * 4 + e]);
      s0 = fmaf(kv.x, a.x, fmaf(kv.y, a.y, s0));
      s1 = fmaf(kv.x, b.x, fmaf(kv.y, b.y, s1));
    }
  }
  float* e = bp.ends + static_cast<size_t>(bh) * 2 * bp.ends_pitch + j;
  e[0] = s0 * bp.scale;
  e[bp.ends_pitch] = s1 * bp.scale;
}

__global__ void __launch_bounds__(128, 2)
    deberta_band_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                        const __grid_constant__ CUtensorMap tmPk, const __grid_constant__ CUtensorMap tmPq,
                        const BandParams bp) {
  const int bh = blockIdx.y;
  if (blockIdx.z == 1) {
    p2c_ends(bp, bh);
    return;
  }
  const int i0 = blockIdx.x * kRows;
  if (i0 >= bp.Lq) return;  // the key side has more blocks

  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_addr);
  const int t = threadIdx.x;
  const int warp = t >> 5;
  const int lane = t & 31;
  const int h = bh % bp.H;
  const int n2k = 2 * bp.k;
  const int nch = (n2k - 1 + kChunk - 1) / kChunk;  // chunks covering m = 1 .. 2k - 1
  const int p_lo = i0 + bp.q_offset;                 // absolute position of row 0
  auto bar = [&](uint32_t i) { return sbase + kOffBar + i * 8; };

  if (t == 0) {
    for (uint32_t i = 0; i < kNBar; ++i) mbar_init(bar(i), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(sbase + kOffBar + kOffSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffBar + kOffSlot);

  // chunk n covers m = 64 n + 1 .. 64 n + 64: Pk rows delta = 2k - m, Pq
  // rows m, and keys j = p_lo + t + m - k for t = 0 .. 127 (table rows or
  // keys outside their tensors load as zeros and feed only values the
  // attention kernel never reads)
  auto load_ops = [&](int n) {  // one thread
    const int m0 = n * kChunk;
    const int jb = p_lo + m0 + 1 - bp.k;
    mbar_arrive_expect_tx(bar(kBarOp), kOpBytes);
    tma_load_3d(sbase + kOffPk, &tmPk, bar(kBarOp), 0, h, n2k - m0 - kChunk);
    tma_load_3d(sbase + kOffPq, &tmPq, bar(kBarOp), 0, h, m0 + 1);
    tma_load_3d(sbase + kOffK, &tmK, bar(kBarOp), 0, jb, bh);
    tma_load_3d(sbase + kOffK + kTile, &tmK, bar(kBarOp), 0, jb + 128, bh);
  };
  if (t == 0) {
    mbar_arrive_expect_tx(bar(kBarQ), kTile);
    tma_load_3d(sbase + kOffQ, &tmQ, bar(kBarQ), 0, i0, bh);
    load_ops(0);
  }

  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  float* stage = reinterpret_cast<float*>(smem + kOffStage);
  uint32_t* outw = reinterpret_cast<uint32_t*>(smem + kOffOut);
  uint32_t* my_row = outw + t * kOutWords;  // row t of the shifted row buffer
  const int sh = (p_lo + t - bp.k) & 7;  // this row's shift
  const bool row_ok = i0 + t < bp.Lq;
  __nv_bfloat16* band_rows = bp.band + (static_cast<size_t>(bh) * bp.Lq + i0) * bp.band_pitch;
  float c_behind = 0.f, c_ahead = 0.f;  // C2P[i][2k - 1], C2P[i][0]
  bool ok = true;
  int loaded = 1;  // chunks whose operands were requested

  for (int n = 0; n < nch; ++n) {
    const int m0 = n * kChunk;
    if (warp == 0) {
      bool w_ok = mbar_wait_warp(bar(kBarOp), n & 1);
      if (w_ok && n == 0) w_ok = mbar_wait_warp(bar(kBarQ), 0);
      tc_fence_after();
      if (w_ok) {
        const uint64_t dq = smem_desc_sw128(sbase + kOffQ, 16, 1024);
        const uint64_t dpk = smem_desc_sw128(sbase + kOffPk, 16, 1024);
        const uint64_t dpq = smem_desc_sw128(sbase + kOffPq, 16, 1024);
        const uint64_t dk0 = smem_desc_sw128(sbase + kOffK, 16, 1024);
        const uint64_t dk1 = smem_desc_sw128(sbase + kOffK + kTile, 16, 1024);
#pragma unroll
        for (int kk = 0; kk < kHeadDim / 16; ++kk) {
          const uint32_t acc = kk > 0 ? 1u : 0u;
          umma_bf16_ss_elect(tmem, dq + 2 * kk, dpk + 2 * kk, kIdesc, acc);
          umma_bf16_ss_elect(tmem + kChunk, dk0 + 2 * kk, dpq + 2 * kk, kIdesc, acc);
          umma_bf16_ss_elect(tmem + 2 * kChunk, dk1 + 2 * kk, dpq + 2 * kk, kIdesc, acc);
        }
        tc_commit_elect(bar(kBarMma));
      }
    }
    // every thread waits (bounded) for the products; a failure anywhere
    // stops the whole CTA at the same chunk
    ok = __syncthreads_and(mbar_wait(bar(kBarMma), n & 1) ? 1 : 0) != 0;
    if (!ok) break;
    tc_fence_after();
    // the operand buffers are free: the next chunk's loads overlap this epilogue
    if (n + 1 < nch) {
      if (t == 0) load_ops(n + 1);
      ++loaded;
    }
    {
      // row positions [0, 8) continue the previous chunk's [64, 72)
#pragma unroll
      for (int w = 0; w < 4; ++w) my_row[w] = n > 0 ? my_row[kChunk / 2 + w] : 0u;
    }
#pragma unroll 1
    for (int u0 = 0; u0 < kChunk; u0 += kSlice) {
      // 1) P2C rows t + u0 .. t + u0 + 31 of the key accumulators, stage row
      //    kappa - u0 for key kappa
      {
        uint32_t va[32], vb[32];
        tmem_ld32(tmem + lane_base + kChunk + u0, va);
        tmem_ld32(tmem + lane_base + 2 * kChunk + u0, vb);
        tmem_ld_wait(va);
        tmem_ld_wait(vb);
        const int ra = warp * 32 + lane - u0;
        const int rb = ra + 128;
        if (ra >= 0) {
#pragma unroll
          for (int e = 0; e < kSlice; ++e) stage[ra * kStagePitch + e] = __uint_as_float(va[e]);
        }
        if (rb < kStageRows) {
#pragma unroll
          for (int e = 0; e < kSlice; ++e) stage[rb * kStagePitch + e] = __uint_as_float(vb[e]);
        }
      }
      __syncthreads();
      // 2) column u = u0 + e of row t: D1[t][63 - u] + D2[t + u][u]
      {
        uint32_t vd[32];
        tmem_ld32(tmem + lane_base + (kChunk - kSlice - u0), vd);
        tmem_ld_wait(vd);
        if (n == 0 && u0 == 0) c_behind = __uint_as_float(vd[31]) * bp.scale;  // m = 1
        const int us = n2k - m0 - 1 - u0;  // slice column of m = 2k (delta(i, j) = 0)
        if (us >= 0 && us < kSlice) {
#pragma unroll
          for (int e = 0; e < kSlice; ++e)
            if (e == us) c_ahead = __uint_as_float(vd[31 - e]) * bp.scale;
        }
        uint32_t w[kSlice / 2];  // bf16 pairs (u0 + 2q, u0 + 2q + 1)
#pragma unroll
        for (int q = 0; q < kSlice / 2; ++q) {
          const int e = 2 * q;
          const float a = (__uint_as_float(vd[31 - e]) + stage[(t + e) * kStagePitch + e]) * bp.scale;
          const float b = (__uint_as_float(vd[30 - e]) + stage[(t + e + 1) * kStagePitch + e + 1]) * bp.scale;
          w[q] = pack_bf16x2(a, b);
        }
        // column u0 sits at row position p0; with p0 odd the pairs straddle
        // words: word (p0 + 1) / 2 + q - 1 takes (u0 + 2q - 1, u0 + 2q) and
        // the two end columns are written as halves
        const int p0 = sh + 1 + u0;
        const bool odd = p0 & 1;
        uint32_t* rw = my_row + (p0 >> 1);
        uint16_t* rh = reinterpret_cast<uint16_t*>(my_row);
        if (odd)
          rh[p0] = static_cast<uint16_t>(w[0] & 0xffffu);
        else
          rw[0] = w[0];
#pragma unroll
        for (int q = 1; q < kSlice / 2; ++q) rw[q] = odd ? __funnelshift_r(w[q - 1], w[q], 16) : w[q];
        if (odd) rh[p0 + kSlice - 1] = static_cast<uint16_t>(w[kSlice / 2 - 1] >> 16);
      }
      __syncthreads();
    }
    // 3) row positions [0, 64) (stored columns m0 .. m0 + 63) are complete:
    //    8 pieces of 16 bytes per row, four rows per warp instruction
#pragma unroll 2
    for (int it = 0; it < kRows * kChunk / 8 / 128; ++it) {
      const int idx = it * 128 + t;
      const int row = idx >> 3;
      const int x = m0 + (idx & 7) * 8;
      if (i0 + row < bp.Lq && x < bp.band_pitch) {
        const uint32_t* src = outw + row * kOutWords + (idx & 7) * 4;
        st_global_v4(band_rows + static_cast<size_t>(row) * bp.band_pitch + x, src[0], src[1], src[2], src[3]);
      }
    }
    if (n == nch - 1 && row_ok && m0 + kChunk < bp.band_pitch)  // the last chunk's overhang [64, 72)
      st_global_v4(band_rows + static_cast<size_t>(t) * bp.band_pitch + m0 + kChunk, my_row[kChunk / 2],
                   my_row[kChunk / 2 + 1], my_row[kChunk / 2 + 2], my_row[kChunk / 2 + 3]);
    tc_fence_before();
    __syncthreads();  // the accumulators and the row buffer are rewritten next
  }
  if (ok && row_ok) {
    float* cc = bp.c2p_const + static_cast<size_t>(bh) * 2 * bp.const_pitch + i0 + t;
    cc[0] = c_behind;
    cc[bp.const_pitch] = c_ahead;
  }
  if (!ok && t == 0 && bp.status) atomicCAS(bp.status, 0, -4);
  if (warp == 0) {
    // no product may still write TMEM and no copy may still write shared
    // memory when the CTA leaves (bounded: after a failure these may not come)
    tc_commit_elect(bar(kBarMma));
    mbar_wait_warp(bar(kBarMma), nch & 1, 100000000ull);
    mbar_wait_warp(bar(kBarOp), (loaded - 1) & 1, 100000000ull);
    mbar_wait_warp(bar(kBarQ), 0, 100000000ull);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    __syncwarp();
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_deberta_band(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmPk,
                                const CUtensorMap& tmPq, const BandParams& bp, cudaStream_t stream) {
  const int bq = (bp.Lq + kRows - 1) / kRows, bk = (bp.Lk + kRows - 1) / kRows;
  dim3 grid(bq > bk ? bq : bk, bp.BH, 2);
  cudaError_t e = cudaFuncSetAttribute(deberta_band_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmem));
  if (e != cudaSuccess) return e;
  deberta_band_kernel<<<grid, 128, kSmem, stream>>>(tmQ, tmK, tmPk, tmPq, bp);
  return cudaGetLastError();
}

}  // namespace relpos
