// txl_prep.cu -- the operands that turn Transformer-XL attention into one
// 128-wide score product ("Relative Position Embeddings, in depth", section
// "Transformer-XL: four terms and two global biases").
//
// The logit of query i (position p) and key j is, scaled by 1/sqrt(d),
//   (q_i + u) . k_j  +  (q_i + v) . W R(p - j)
// with R(t) the fixed sinusoidal encoding (R[2m] = sin(w_m t),
// R[2m+1] = cos(w_m t), w_m = 10000^(-2m/d)) and W the head's key projection
// of it. With a = W^T (q_i + v) the position term is a . R(p - j), and the
// angle-difference identities split it into a query part and a key part:
//   a . R(p - j) = sum_m  cos(w_m j) (a_2m sin(w_m p) + a_2m+1 cos(w_m p))
//                       + sin(w_m j) (a_2m+1 sin(w_m p) - a_2m cos(w_m p)).
// So the whole logit is one dot product of 128-vectors,
//   [q_i + u | a rotated by w p] . [k_j | (cos w_m j, sin w_m j)_m],
// which the fused kernel computes on the tensor cores like Q K^T. Nothing
// indexed by the offset is formed: the pages' skew over an L x (L + mem)
// matrix is not needed.
//
// This kernel writes the query side Q2 [BH, Lq, 128] (bf16) and the key
// sinusoid table S [Lk, 64] (bf16, the same for every head). Query blocks:
// 128 rows of one head per CTA; each thread stages its row of q + v (bf16)
// as the A operand of one tcgen05 product a = (Q + v) W (M128 N64 K64, W as
// an MN-major bf16 operand in shared memory, fp32 accumulator in TMEM),
// then takes its row of a out of TMEM, rotates it by its angles and stores
// both halves. Key blocks (blockIdx.y == BH): one thread per key.

#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"
#include "relpos_common.cuh"
#include "relpos_internal.h"

namespace relpos {
namespace {

constexpr int kPrepThreads = 128;
constexpr int kRowsPerBlock = kPrepThreads;
constexpr uint32_t kIdescAW = idesc_bf16_f32(128, kHeadDim, 0, 1);  // A K-major, B MN-major

__global__ void __launch_bounds__(kPrepThreads) txl_prep_kernel(const TxlParams p) {
  // A: 128 rows x 128 B (q + v, bf16); B: 64 rows (e) x 128 B (W[e][0..63], bf16);
  // both 128-byte swizzled, 1024-byte aligned
  __shared__ __align__(1024) uint8_t a_s[128 * 128];
  __shared__ __align__(1024) uint8_t w_s[64 * 128];
  __shared__ __align__(8) uint64_t bar;
  __shared__ uint32_t tmem_slot;
  const int tid = threadIdx.x;
  if (static_cast<int>(blockIdx.y) == p.BH) {
    griddep_wait();
    // key sinusoid table: row j = (cos w_m j, sin w_m j) for m = 0 .. 31
    const int j = blockIdx.x * kPrepThreads + tid;
    if (j >= p.Lk) return;
    uint4* dst = reinterpret_cast<uint4*>(p.Ksin + static_cast<size_t>(j) * kHeadDim);
    const float fj = static_cast<float>(j);
#pragma unroll
    for (int c = 0; c < 8; ++c) {  // 8 components (4 frequencies) per 16-byte piece
      uint32_t w4[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float sn, cs;
        sincosf(fj * p.omega[4 * c + e], &sn, &cs);
        w4[e] = pack_bf16x2(cs, sn);
      }
      dst[c] = make_uint4(w4[0], w4[1], w4[2], w4[3]);
    }
    return;
  }
  const int bh = blockIdx.y;
  const int h = bh % p.H;
  const int row0 = blockIdx.x * kRowsPerBlock;
  if (row0 >= p.Lq) return;  // uniform over the CTA
  const int warp = tid >> 5;
  if (tid == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(&tmem_slot), 64);
    tmem_relinquish();
  }
  griddep_wait();
  // W (fp32, [e][f]) to bf16: row e of the MN-major operand holds f = 0 .. 63
  {
    const float4* wsrc = reinterpret_cast<const float4*>(p.W + static_cast<size_t>(h) * kHeadDim * kHeadDim);
    for (int i = tid; i < kHeadDim * kHeadDim / 8; i += kPrepThreads) {  // 8 values (16 B) each
      const int e = i >> 3, ch = i & 7;
      const float4 x0 = __ldg(wsrc + 2 * i), x1 = __ldg(wsrc + 2 * i + 1);
      const uint4 v4 = make_uint4(pack_bf16x2(x0.x, x0.y), pack_bf16x2(x0.z, x0.w), pack_bf16x2(x1.x, x1.y),
                                  pack_bf16x2(x1.z, x1.w));
      *reinterpret_cast<uint4*>(w_s + e * 128 + ((ch ^ (e & 7)) << 4)) = v4;
    }
  }
  const int row = row0 + tid;
  const bool row_ok = row < p.Lq;
  const size_t qrow = static_cast<size_t>(bh) * p.Lq + (row_ok ? row : row0);
  const float* u = p.uv + static_cast<size_t>(h) * kHeadDim;
  const float* v = p.uv + (static_cast<size_t>(p.H) + h) * kHeadDim;
  uint4* dst = reinterpret_cast<uint4*>(p.Q2 + qrow * (2 * kHeadDim));
  // content half q + u to global; q + v (bf16) to the A operand (zero rows past Lq)
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.Q + qrow * kHeadDim);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 u4 = __ldg(src + c);
      const uint32_t w4[4] = {u4.x, u4.y, u4.z, u4.w};
      uint32_t qu[4], qv[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
        const int k = 8 * c + 2 * e;
        qu[e] = pack_bf16x2(f.x + __ldg(u + k), f.y + __ldg(u + k + 1));
        qv[e] = row_ok ? pack_bf16x2(f.x + __ldg(v + k), f.y + __ldg(v + k + 1)) : 0u;
      }
      if (row_ok) dst[c] = make_uint4(qu[0], qu[1], qu[2], qu[3]);
      *reinterpret_cast<uint4*>(a_s + tid * 128 + ((c ^ (tid & 7)) << 4)) = make_uint4(qv[0], qv[1], qv[2], qv[3]);
    }
  }
  fence_async_smem();  // the operands' generic writes, visible to the tensor core
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = tmem_slot;
  if (tid == 0) {
    const uint64_t da = smem_desc_sw128(smem_u32(a_s), 16, 1024);
    const uint64_t dw = smem_desc_sw128(smem_u32(w_s), 8192, 1024);
#pragma unroll
    for (int kk = 0; kk < kHeadDim / 16; ++kk)  // K-step of 16 e: 32 B of A's rows, 2 row groups of W
      umma_bf16_ss(tmem, da + 2 * kk, dw + 128 * kk, kIdescAW, kk > 0 ? 1u : 0u);
    tc_commit(smem_u32(&bar));
  }
  const bool ok = mbar_wait(smem_u32(&bar), 0);
  tc_fence_after();
  // a of this row (TMEM lane tid), rotated by the angles w_m p
  const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
  const float pos = static_cast<float>(row + p.q_offset);
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t r[32];
    tmem_ld32(tmem + lane_base + 32 * half, r);
    tmem_ld_wait(r);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      uint32_t rot[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const int mm = 4 * c + e;          // pair within the half
        const int m = 16 * half + mm;      // frequency index
        float sn, cs;
        sincosf(pos * p.omega[m], &sn, &cs);
        const float a0 = __uint_as_float(r[2 * mm]), a1 = __uint_as_float(r[2 * mm + 1]);
        rot[e] = pack_bf16x2(fmaf(a0, sn, a1 * cs), fmaf(a1, sn, -a0 * cs));
      }
      if (row_ok && ok) dst[8 + 4 * half + c] = make_uint4(rot[0], rot[1], rot[2], rot[3]);
    }
  }
  if (!ok && tid == 0 && p.status) atomicCAS(p.status, 0, -4);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, 64);
  }
}

}  // namespace

cudaError_t launch_txl_prep(const TxlParams& p, cudaStream_t stream) {
  const int qblocks = (p.Lq + kRowsPerBlock - 1) / kRowsPerBlock;
  const int kblocks = (p.Lk + kPrepThreads - 1) / kPrepThreads;
  const int gx = qblocks > kblocks ? qblocks : kblocks;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(gx, p.BH + 1);
  cfg.blockDim = dim3(kPrepThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, txl_prep_kernel, p);
}

}  // namespace relpos
