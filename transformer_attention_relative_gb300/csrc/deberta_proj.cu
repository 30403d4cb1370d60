// deberta_proj.cu -- the relative-position products of DeBERTa attention:
//   C2P[bh][i][r] = s * q_i . Pk[r][h]   and   P2C[bh][j][r] = s * k_j . Pq[r][h]
// for every table row r in [0, 2k) ("Relative Position Embeddings, in depth",
// section "DeBERTa: disentangled content and position"; the table index is
// delta of "DeBERTa > Relative Position Encoding", "The Relative Position
// Formula"). This is the form the pages call workable for relative keys
// ("Shaw et al."): the rows times the 2k-row table, an L x 2k matrix, which
// the attention kernel then reads by clipped offset. s is the softmax scale
// times log2(e), so the attention kernel adds the values to its log2-domain
// logits directly. For P2C the two end columns (r = 0 and r = 2k - 1, the
// values every key takes once the offset saturates) are also written in fp32
// as ends[bh][0 | 1][j].
//
// One launch computes both products (grid z: C2P, P2C). One CTA (128
// threads, four per SM) per 128-row tile of one head: TMA brings the Q (or
// K) tile and 64-row chunks of the table (two buffers); tcgen05.mma M128 N64
// K16 accumulates a chunk into one half of a 128-column TMEM allocation while
// the four warps drain the other half. Each warp stages its 32 rows of a
// chunk in shared memory (128-byte rows, 16-byte pieces swizzled by row) and
// stores them back four whole row segments per instruction.

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"
#include "relpos_common.cuh"
#include "relpos_internal.h"

namespace relpos {
namespace {

constexpr int kRows = 128;
constexpr int kChunk = 64;  // table rows per MMA group (N)
constexpr uint32_t kATile = kRows * kHeadDim * 2;   // 16 KB
constexpr uint32_t kBTile = kChunk * kHeadDim * 2;  // 16 KB
constexpr uint32_t kWarpStage = 32 * kChunk * 2;    // 32 rows x kChunk bf16
constexpr int kLanesPerRow = kChunk / 8;            // 16-byte pieces of a staged row
constexpr int kRowsPerStore = 32 / kLanesPerRow;    // rows one warp store covers
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kATile;                  // two chunk buffers
constexpr uint32_t kOffStage = kOffB + 2 * kBTile;  // four warps' staging
constexpr uint32_t kOffBar = kOffStage + 4 * kWarpStage;
constexpr uint32_t kSmem = 1024 + kOffBar + 128;
constexpr uint32_t kIdesc = idesc_bf16_f32(kRows, kChunk, 0, 0);
constexpr uint32_t kTmemCols = 2 * kChunk;

enum : uint32_t { kBarA = 0, kBarB = 1, kBarDone = 3, kBarFinal = 5, kNBar = 6 };
constexpr uint32_t kOffSlot = kNBar * 8;

__global__ void __launch_bounds__(128, 4)
    deberta_proj_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmPk,
                        const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmPq,
                        const ProjParams pp) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_addr);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int t = threadIdx.x;
  const int side = blockIdx.z;  // 0: C2P, 1: P2C
  const int L = pp.L[side];
  const int i0 = blockIdx.x * kRows;
  if (i0 >= L) return;  // the other side has more rows
  const bool ends = side == 1 && pp.ends != nullptr;
  const CUtensorMap* tmA = side ? &tmK : &tmQ;
  const CUtensorMap* tmP = side ? &tmPq : &tmPk;
  __nv_bfloat16* out = pp.out[side];
  const int bh = blockIdx.y;
  const int h = bh % pp.H;
  const int n2k = 2 * pp.k;
  const int nch = (n2k + kChunk - 1) / kChunk;
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

  auto load_b = [&](int c) {  // warp 0
    const uint32_t b = c & 1;
    mbar_arrive_expect_tx_elect(bar(kBarB + b), kBTile);
    tma_load_3d_elect(sbase + kOffB + b * kBTile, tmP, bar(kBarB + b), 0, h, c * kChunk);
  };
  bool ok = true;
  auto issue = [&](int c) {  // warp 0
    const uint32_t b = c & 1;
    ok = ok && mbar_wait_warp(bar(kBarB + b), (c >> 1) & 1);
    tc_fence_after();
    if (!ok) return;
    const uint64_t da = smem_desc_sw128(sbase + kOffA, 16, 1024);
    const uint64_t db = smem_desc_sw128(sbase + kOffB + b * kBTile, 16, 1024);
#pragma unroll
    for (int kk = 0; kk < kHeadDim / 16; ++kk)
      umma_bf16_ss_elect(tmem + b * kChunk, da + 2 * kk, db + 2 * kk, kIdesc, kk > 0 ? 1u : 0u);
    tc_commit_elect(bar(kBarDone + b));
  };

  if (warp == 0) {
    mbar_arrive_expect_tx_elect(bar(kBarA), kATile);
    tma_load_3d_elect(sbase + kOffA, tmA, bar(kBarA), 0, i0, bh);
    load_b(0);
    if (nch > 1) load_b(1);
    ok = mbar_wait_warp(bar(kBarA), 0);
    issue(0);
  }
  const int row = i0 + t;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const bool vec_ok = (n2k & 7) == 0;  // 16-byte aligned rows: staged, coalesced stores
  const uint32_t stage = sbase + kOffStage + warp * kWarpStage;
  __nv_bfloat16* dst_row = out + (static_cast<size_t>(bh) * L + (row < L ? row : 0)) * n2k;
  for (int c = 0; c < nch; ++c) {
    if (warp == 0 && c + 1 < nch) issue(c + 1);
    const uint32_t b = c & 1;
    const bool good = mbar_wait_warp(bar(kBarDone + b), (c >> 1) & 1);
    if (!good) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (warp == 0 && c + 2 < nch) load_b(c + 2);  // buffer b has been read
#pragma unroll 1
    for (int q = 0; q < kChunk / 32; ++q) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_base + b * kChunk + q * 32, v);
      tmem_ld_wait(v);
      const int col0 = c * kChunk + q * 32;
      float f[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v[e]) * pp.scale;
      if (ends) {
        if (row < L) {
          if (col0 == 0) pp.ends[(static_cast<size_t>(bh) * 2 + 0) * pp.ends_pitch + row] = f[0];
          const int last = n2k - 1 - col0;
          if (last >= 0 && last < 32) {
#pragma unroll
            for (int e = 0; e < 32; ++e)
              if (e == last) pp.ends[(static_cast<size_t>(bh) * 2 + 1) * pp.ends_pitch + row] = f[e];
          }
        }
      }
      if (vec_ok) {
        // chunk cc (8 columns) of this lane's row: box cc / 8, 16-byte slot
        // (cc % 8) ^ (row % 8)
#pragma unroll
        for (int m = 0; m < 4; ++m) {
          const int cc = q * 4 + m;
          const uint32_t a = stage + (cc >> 3) * (32u * 128u) + lane * 128u + (((cc & 7) ^ (lane & 7)) << 4);
          st_shared_v4(a, pack_bf16x2(f[8 * m], f[8 * m + 1]), pack_bf16x2(f[8 * m + 2], f[8 * m + 3]),
                       pack_bf16x2(f[8 * m + 4], f[8 * m + 5]), pack_bf16x2(f[8 * m + 6], f[8 * m + 7]));
        }
      } else if (row < L) {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (col0 + e < n2k) dst_row[col0 + e] = __float2bfloat16_rn(f[e]);
      }
    }
    if (vec_ok) {
      // kRowsPerStore whole row segments per store instruction
      __syncwarp();
#pragma unroll 4
      for (int it = 0; it < 32 / kRowsPerStore; ++it) {
        const int r = kRowsPerStore * it + lane / kLanesPerRow;
        const int cc = lane % kLanesPerRow;
        const int grow = i0 + warp * 32 + r;
        const int gcol = c * kChunk + cc * 8;
        uint32_t w0, w1, w2, w3;
        ld_shared_v4(stage + (cc >> 3) * (32u * 128u) + r * 128u + (((cc & 7) ^ (r & 7)) << 4), w0, w1, w2, w3);
        if (grow < L && gcol < n2k)
          st_global_v4(out + (static_cast<size_t>(bh) * L + grow) * n2k + gcol, w0, w1, w2, w3);
      }
      __syncwarp();  // the staging is rewritten by the next chunk
    }
    tc_fence_before();
    __syncthreads();  // this TMEM half may be overwritten by chunk c + 2
    tc_fence_after();
  }
  if (!ok && t == 0 && pp.status) atomicCAS(pp.status, 0, -4);
  if (warp == 0) {
    // every issued product has finished, and no copy is in flight
    tc_commit_elect(bar(kBarFinal));
    mbar_wait_warp(bar(kBarFinal), 0, 100000000ull);
    for (int c = (nch > 2 ? nch - 2 : 0); c < nch; ++c)
      mbar_wait_warp(bar(kBarB + (c & 1)), (c >> 1) & 1, 100000000ull);
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

cudaError_t launch_deberta_proj(const CUtensorMap& tmQ, const CUtensorMap& tmPk, const CUtensorMap& tmK,
                                const CUtensorMap& tmPq, const ProjParams& pp, cudaStream_t stream) {
  const int rows = pp.L[0] > pp.L[1] ? pp.L[0] : pp.L[1];
  dim3 grid((rows + kRows - 1) / kRows, pp.BH, 2);
  cudaError_t e = cudaFuncSetAttribute(deberta_proj_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(kSmem));
  if (e != cudaSuccess) return e;
  deberta_proj_kernel<<<grid, 128, kSmem, stream>>>(tmQ, tmPk, tmK, tmPq, pp);
  return cudaGetLastError();
}

}  // namespace relpos
