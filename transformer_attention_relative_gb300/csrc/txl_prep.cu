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
// 128 threads, 32 rows, four threads per row, each forming 16 of the 64
// components of a (the head's W staged in shared memory). Key blocks
// (blockIdx.y == BH): one thread per key.

#include <cuda_bf16.h>

#include <cstdint>

#include "ptx.cuh"
#include "relpos_common.cuh"
#include "relpos_internal.h"

namespace relpos {
namespace {

constexpr int kPrepThreads = 128;
constexpr int kRowsPerBlock = kPrepThreads / 4;

__global__ void __launch_bounds__(kPrepThreads) txl_prep_kernel(const TxlParams p) {
  __shared__ __align__(16) float w_s[kHeadDim * kHeadDim];  // W[e][f] of this head
  __shared__ __align__(16) float wv_s[kHeadDim];            // W^T v
  griddep_wait();
  const int tid = threadIdx.x;
  if (static_cast<int>(blockIdx.y) == p.BH) {
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
  if (row0 >= p.Lq) return;
  {
    const float4* src = reinterpret_cast<const float4*>(p.W + static_cast<size_t>(h) * kHeadDim * kHeadDim);
    float4* dst = reinterpret_cast<float4*>(w_s);
    for (int i = tid; i < kHeadDim * kHeadDim / 4; i += kPrepThreads) dst[i] = __ldg(src + i);
  }
  __syncthreads();
  if (tid < kHeadDim) {  // W^T v, added to every row's a
    const float* v = p.uv + (static_cast<size_t>(p.H) + h) * kHeadDim;
    float acc = 0.f;
    for (int e = 0; e < kHeadDim; ++e) acc = fmaf(__ldg(v + e), w_s[e * kHeadDim + tid], acc);
    wv_s[tid] = acc;
  }
  __syncthreads();
  const int r = tid >> 2;   // row within the block
  const int g = tid & 3;    // components 16 g .. 16 g + 15
  const int row = row0 + r;
  if (row >= p.Lq) return;
  const size_t qrow = static_cast<size_t>(bh) * p.Lq + row;
  float q[kHeadDim];
  {
    const uint4* src = reinterpret_cast<const uint4*>(p.Q + qrow * kHeadDim);
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      const uint4 u4 = __ldg(src + c);
      const uint32_t w4[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
        q[8 * c + 2 * e] = f.x;
        q[8 * c + 2 * e + 1] = f.y;
      }
    }
  }
  // a_f = sum_e q_e W[e][f] + (W^T v)_f for this thread's 16 components
  float a[16];
#pragma unroll
  for (int f = 0; f < 16; ++f) a[f] = wv_s[16 * g + f];
#pragma unroll
  for (int e = 0; e < kHeadDim; ++e) {
    const float4* wr = reinterpret_cast<const float4*>(w_s + e * kHeadDim + 16 * g);
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const float4 w4 = wr[c];
      a[4 * c] = fmaf(q[e], w4.x, a[4 * c]);
      a[4 * c + 1] = fmaf(q[e], w4.y, a[4 * c + 1]);
      a[4 * c + 2] = fmaf(q[e], w4.z, a[4 * c + 2]);
      a[4 * c + 3] = fmaf(q[e], w4.w, a[4 * c + 3]);
    }
  }
  // the query half of the position product: a rotated by the angles w_m p
  const float pos = static_cast<float>(row + p.q_offset);
  uint32_t rot[8];
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    float sn, cs;
    sincosf(pos * p.omega[8 * g + m], &sn, &cs);
    const float a0 = a[2 * m], a1 = a[2 * m + 1];
    rot[m] = pack_bf16x2(fmaf(a0, sn, a1 * cs), fmaf(a1, sn, -a0 * cs));
  }
  // the content half: q + u, components 16 g .. 16 g + 15 (reloaded: q[]
  // is indexed by constants only, so it stays in registers)
  const float* u = p.uv + static_cast<size_t>(h) * kHeadDim + 16 * g;
  const uint4* qg = reinterpret_cast<const uint4*>(p.Q + qrow * kHeadDim) + 2 * g;
  uint32_t qu[8];
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    const uint4 u4 = __ldg(qg + c);
    const uint32_t w4[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w4[e]));
      qu[4 * c + e] = pack_bf16x2(f.x + __ldg(u + 8 * c + 2 * e), f.y + __ldg(u + 8 * c + 2 * e + 1));
    }
  }
  uint4* dst = reinterpret_cast<uint4*>(p.Q2 + qrow * (2 * kHeadDim));
  dst[2 * g] = make_uint4(qu[0], qu[1], qu[2], qu[3]);
  dst[2 * g + 1] = make_uint4(qu[4], qu[5], qu[6], qu[7]);
  dst[8 + 2 * g] = make_uint4(rot[0], rot[1], rot[2], rot[3]);
  dst[8 + 2 * g + 1] = make_uint4(rot[4], rot[5], rot[6], rot[7]);
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
