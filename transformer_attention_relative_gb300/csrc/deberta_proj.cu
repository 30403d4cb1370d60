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
// One CTA (128 threads) per 128-row tile of one head: TMA brings the Q (or K)
// tile and 256-row chunks of the table (two buffers); tcgen05.mma M128 N256
// K16 accumulates a chunk into one half of TMEM while the four warps drain
// the other half to global memory (bf16).

#include <cuda.h>
#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"
#include "relpos_common.cuh"
#include "relpos_internal.h"

namespace relpos {
namespace {

constexpr int kRows = 128;
constexpr int kChunk = 256;  // table rows per MMA group (N)
constexpr uint32_t kATile = kRows * kHeadDim * 2;   // 16 KB
constexpr uint32_t kBTile = kChunk * kHeadDim * 2;  // 32 KB
constexpr uint32_t kOffA = 0;
constexpr uint32_t kOffB = kATile;                  // two chunk buffers
constexpr uint32_t kOffBar = kOffB + 2 * kBTile;
constexpr uint32_t kSmem = 1024 + kOffBar + 128;
constexpr uint32_t kIdesc = idesc_bf16_f32(kRows, kChunk, 0, 0);

enum : uint32_t { kBarA = 0, kBarB = 1, kBarDone = 3, kBarFinal = 5, kNBar = 6 };
constexpr uint32_t kOffSlot = kNBar * 8;

template <bool ENDS>
__global__ void __launch_bounds__(128, 1)
    deberta_proj_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmP,
                        const ProjParams pp) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  const uint32_t sbase = (raw_addr + 1023u) & ~1023u;
  uint8_t* smem = smem_raw + (sbase - raw_addr);
  const int warp = threadIdx.x >> 5;
  const int t = threadIdx.x;
  const int i0 = blockIdx.x * kRows;
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
    tmem_alloc(sbase + kOffBar + kOffSlot, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *reinterpret_cast<volatile uint32_t*>(smem + kOffBar + kOffSlot);

  auto load_b = [&](int c) {  // warp 0
    const uint32_t b = c & 1;
    mbar_arrive_expect_tx_elect(bar(kBarB + b), kBTile);
    tma_load_3d_elect(sbase + kOffB + b * kBTile, &tmP, bar(kBarB + b), 0, h, c * kChunk);
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
    tma_load_3d_elect(sbase + kOffA, &tmA, bar(kBarA), 0, i0, bh);
    load_b(0);
    if (nch > 1) load_b(1);
    ok = mbar_wait_warp(bar(kBarA), 0);
    issue(0);
  }
  const int row = i0 + t;
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  __nv_bfloat16* dst_row = pp.out + (static_cast<size_t>(bh) * pp.L + (row < pp.L ? row : 0)) * n2k;
  const bool vec_ok = (n2k & 7) == 0;  // 16-byte aligned row segments
  for (int c = 0; c < nch; ++c) {
    if (warp == 0 && c + 1 < nch) issue(c + 1);
    const uint32_t b = c & 1;
    bool good = mbar_wait(bar(kBarDone + b), (c >> 1) & 1);
    good = __all_sync(0xffffffffu, good);
    if (!good) {
      ok = false;
      break;
    }
    tc_fence_after();
    if (warp == 0 && c + 2 < nch) load_b(c + 2);  // buffer b has been read
    __syncwarp();
#pragma unroll 1
    for (int q = 0; q < kChunk / 32; ++q) {
      uint32_t v[32];
      tmem_ld32(tmem + lane_base + b * kChunk + q * 32, v);
      tmem_ld_wait(v);
      const int col0 = c * kChunk + q * 32;
      if (row >= pp.L || col0 >= n2k) continue;
      float f[32];
#pragma unroll
      for (int e = 0; e < 32; ++e) f[e] = __uint_as_float(v[e]) * pp.scale;
      if constexpr (ENDS) {
        if (col0 == 0) pp.ends[(static_cast<size_t>(bh) * 2 + 0) * pp.ends_pitch + row] = f[0];
        const int last = n2k - 1 - col0;
        if (last >= 0 && last < 32) {
#pragma unroll
          for (int e = 0; e < 32; ++e)
            if (e == last) pp.ends[(static_cast<size_t>(bh) * 2 + 1) * pp.ends_pitch + row] = f[e];
        }
      }
      if (vec_ok && col0 + 32 <= n2k) {
#pragma unroll
        for (int e = 0; e < 32; e += 8)
          st_global_v4(dst_row + col0 + e, pack_bf16x2(f[e], f[e + 1]), pack_bf16x2(f[e + 2], f[e + 3]),
                       pack_bf16x2(f[e + 4], f[e + 5]), pack_bf16x2(f[e + 6], f[e + 7]));
      } else {
#pragma unroll
        for (int e = 0; e < 32; ++e)
          if (col0 + e < n2k) dst_row[col0 + e] = __float2bfloat16_rn(f[e]);
      }
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
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

cudaError_t launch_deberta_proj(bool ends, const CUtensorMap& tmA, const CUtensorMap& tmP,
                                const ProjParams& pp, cudaStream_t stream) {
  dim3 grid((pp.L + kRows - 1) / kRows, pp.BH);
  auto kern = ends ? deberta_proj_kernel<true> : deberta_proj_kernel<false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmem));
  if (e != cudaSuccess) return e;
  kern<<<grid, 128, kSmem, stream>>>(tmA, tmP, pp);
  return cudaGetLastError();
}

}  // namespace relpos
