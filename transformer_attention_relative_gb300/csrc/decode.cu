// decode.cu -- T5-bias (and, over explicit key positions, ALiBi) attention
// for a few query rows against a long key cache (cached decoding: "T5
// Relative-Position Bias", cached-decoder example; "Relative Position
// Embeddings, in depth", "Kernels and the KV cache"). With one query row per (batch, head) the work is a stream over K
// and V (about one flop per byte), so it runs on CUDA cores, split over key
// chunks so that every SM keeps many 16-byte loads in flight, followed by a
// small combine of the per-chunk (max, sum, partial output).
//
// Query row i sits at absolute position i + q_offset; its offsets to key j
// are j - (i + q_offset), bucketed by the same device generator the fused
// kernel uses.

#include <cuda_bf16.h>

#include <algorithm>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/relpos_attn.h"
#include "ptx.cuh"
#include "relpos_common.cuh"
#include "relpos_internal.h"

namespace relpos {
namespace {

constexpr int kDecThreads = 128;    // 16 groups of 8 threads; a group reads one 128-byte key row
constexpr int kDecChunk = 256;      // keys per CTA
constexpr int kKeysPerThread = kDecChunk / 16;

RP_DEVI void bf16x8_to_f32(const uint4& u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[e]));
    f[2 * e] = v.x;
    f[2 * e + 1] = v.y;
  }
}

__global__ void __launch_bounds__(kDecThreads, 3) relpos_decode_partial_kernel(const DecodeParams p) {
  const int chunk = blockIdx.x;
  const int qi = blockIdx.y;
  const int bh = blockIdx.z;
  const int h = bh % p.H;
  const int tid = threadIdx.x;
  const int grp = tid >> 3;  // 0..15: key row within a 16-row slab
  const int sl = tid & 7;    // 8-dim slice of the head dimension
  const int warp = tid >> 5;

  __shared__ float bias_s[kDecChunk];  // log2-scaled bias of each key of the chunk
  __shared__ float red_s[4];
  __shared__ float o_s[4][kHeadDim];

  griddep_wait();  // the previous kernel of the stream has completed
  // ALiBi (t5_R < 0): bias holds the heads' slopes, and an offset's bias is
  // -slope |offset| (log2 units below), with no saturation
  const bool alibi = p.t5_R < 0;
  const float slope2 = alibi ? __ldg(p.bias + h) * kLog2e : 0.f;
  const int pos = qi + p.q_offset;
  const int jb = chunk * kDecChunk;
  // explicit key positions (a cache that evicted keys): visibility follows
  // the positions, not the key index
  const int* kpos = p.key_pos ? p.key_pos + static_cast<size_t>(bh) * p.Lk : nullptr;
  int je = min(p.Lk, jb + kDecChunk);
  if (p.causal && !kpos) je = min(je, pos + 1);

  const size_t row_out = static_cast<size_t>(bh) * p.Lq + qi;
  float* po = p.part_o + (row_out * p.nchunks + chunk) * kHeadDim;
  float* pml = p.part_ml + (row_out * p.nchunks + chunk) * 2;

  if (jb >= je) {  // nothing visible in this chunk
    if (tid < kHeadDim) po[tid] = 0.f;
    if (tid == 0) {
      pml[0] = -INFINITY;
      pml[1] = 0.f;
    }
    return;
  }

  // start the chunk's K and V rows towards L2 now: the bias setup below (for
  // explicit positions a dependent position load, bucket and gather per key)
  // then overlaps their DRAM latency, and no register is held meanwhile
  {
    const char* kr = reinterpret_cast<const char*>(p.K + (static_cast<size_t>(bh) * p.Lk + jb) * kHeadDim);
    const char* vr = reinterpret_cast<const char*>(p.V + (static_cast<size_t>(bh) * p.Lk + jb) * kHeadDim);
    for (int r = tid; r < je - jb; r += kDecThreads) {
      prefetch_l2(kr + static_cast<size_t>(r) * kHeadDim * 2);
      prefetch_l2(vr + static_cast<size_t>(r) * kHeadDim * 2);
    }
  }
  // The chunk's offsets run from jb - pos to je - 1 - pos. Past the saturation
  // distance R every key of a side takes that side's last bucket, so a chunk
  // lying wholly beyond R needs one bias; otherwise each key's bias is looked
  // up once here rather than by every thread that shares the key.
  const int rel_first = jb - pos, rel_last = je - 1 - pos;
  const bool sat_l = !kpos && !alibi && rel_last <= -p.t5_R;
  const bool sat_r = !kpos && !alibi && p.t5.bidir && rel_first >= p.t5_R;
  float bias_const = 0.f;
  if (sat_l || sat_r) {
    bias_const = __ldg(p.bias + t5_bucket_dev(sat_l ? -p.t5_R : p.t5_R, p.t5) * p.H + h) * kLog2e;
  } else if (kpos) {
    // per key: the bias of its own offset, -inf for a key after the query.
    // A thread's two keys are written out side by side so that both position
    // loads, then both table loads, are in flight together.
    static_assert(kDecChunk == 2 * kDecThreads, "two keys per thread");
    const int r0 = tid, r1 = tid + kDecThreads;
    const bool in0 = jb + r0 < je, in1 = jb + r1 < je;
    const int rel0 = (in0 ? __ldg(kpos + jb + r0) : pos) - pos;
    const int rel1 = (in1 ? __ldg(kpos + jb + r1) : pos) - pos;
    const bool vis0 = in0 && (!p.causal || rel0 <= 0);
    const bool vis1 = in1 && (!p.causal || rel1 <= 0);
    float b0 = 0.f, b1 = 0.f;
    if (alibi) {
      b0 = -slope2 * fabsf(static_cast<float>(rel0));
      b1 = -slope2 * fabsf(static_cast<float>(rel1));
    } else {
      b0 = vis0 ? __ldg(p.bias + t5_bucket_dev(rel0, p.t5) * p.H + h) * kLog2e : 0.f;
      b1 = vis1 ? __ldg(p.bias + t5_bucket_dev(rel1, p.t5) * p.H + h) * kLog2e : 0.f;
    }
    bias_s[r0] = vis0 ? b0 : -INFINITY;
    bias_s[r1] = vis1 ? b1 : -INFINITY;
  } else {
    for (int r = tid; r < kDecChunk; r += kDecThreads)
      bias_s[r] = alibi ? -slope2 * fabsf(static_cast<float>(jb + r - pos))
                        : __ldg(p.bias + t5_bucket_dev(jb + r - pos, p.t5) * p.H + h) * kLog2e;
  }
  const bool sat = sat_l || sat_r;

  // issue every K and V load of this thread first
  const uint4* kbase = reinterpret_cast<const uint4*>(p.K + static_cast<size_t>(bh) * p.Lk * kHeadDim);
  const uint4* vbase = reinterpret_cast<const uint4*>(p.V + static_cast<size_t>(bh) * p.Lk * kHeadDim);
  uint4 kv[kKeysPerThread], vv[kKeysPerThread];
#pragma unroll
  for (int r = 0; r < kKeysPerThread; ++r) {
    const int j = jb + grp + 16 * r;
    if (j < je) {
      kv[r] = __ldg(kbase + static_cast<size_t>(j) * 8 + sl);
      vv[r] = __ldg(vbase + static_cast<size_t>(j) * 8 + sl);
    } else {
      kv[r] = make_uint4(0, 0, 0, 0);
      vv[r] = make_uint4(0, 0, 0, 0);
    }
  }
  float qf[8];
  {
    const uint4 qv = __ldg(reinterpret_cast<const uint4*>(p.Q + row_out * kHeadDim) + sl);
    bf16x8_to_f32(qv, qf);
  }
  __syncthreads();  // bias_s

  float s[kKeysPerThread];
  float mx = -INFINITY;
#pragma unroll
  for (int r = 0; r < kKeysPerThread; ++r) {
    float kf[8];
    bf16x8_to_f32(kv[r], kf);
    float acc = 0.f;
#pragma unroll
    for (int e = 0; e < 8; ++e) acc = fmaf(qf[e], kf[e], acc);
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    const int j = jb + grp + 16 * r;
    const float bias = sat ? bias_const : bias_s[grp + 16 * r];
    s[r] = (j < je) ? fmaf(acc, p.scale_log2, bias) : -INFINITY;
    mx = fmaxf(mx, s[r]);
  }
  // max over the CTA (groups within a warp differ in lanes 8, 16)
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
  if ((tid & 31) == 0) red_s[warp] = mx;
  __syncthreads();
  mx = fmaxf(fmaxf(red_s[0], red_s[1]), fmaxf(red_s[2], red_s[3]));
  __syncthreads();
  if (mx == -INFINITY) {  // every key of the chunk masked by its position
    if (tid < kHeadDim) po[tid] = 0.f;
    if (tid == 0) {
      pml[0] = -INFINITY;
      pml[1] = 0.f;
    }
    return;
  }

  float sum = 0.f;
  float o[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
  for (int r = 0; r < kKeysPerThread; ++r) {
    const float pr = ex2_approx(s[r] - mx);
    sum += pr;
    float vf[8];
    bf16x8_to_f32(vv[r], vf);
#pragma unroll
    for (int e = 0; e < 8; ++e) o[e] = fmaf(pr, vf[e], o[e]);
  }
  sum += __shfl_xor_sync(0xffffffffu, sum, 8);
  sum += __shfl_xor_sync(0xffffffffu, sum, 16);
#pragma unroll
  for (int e = 0; e < 8; ++e) {
    o[e] += __shfl_xor_sync(0xffffffffu, o[e], 8);
    o[e] += __shfl_xor_sync(0xffffffffu, o[e], 16);
  }
  if ((tid & 31) < 8) {
#pragma unroll
    for (int e = 0; e < 8; ++e) o_s[warp][sl * 8 + e] = o[e];
  }
  if ((tid & 31) == 0) red_s[warp] = sum;
  __syncthreads();
  if (tid < kHeadDim) po[tid] = (o_s[0][tid] + o_s[1][tid]) + (o_s[2][tid] + o_s[3][tid]);
  if (tid == 0) {
    pml[0] = mx;
    pml[1] = (red_s[0] + red_s[1]) + (red_s[2] + red_s[3]);
  }
  griddep_launch_dependents();  // the combine may be scheduled now
}

// one warp per (row, 64 dims): merge the per-chunk partials
__global__ void __launch_bounds__(64) relpos_decode_combine_kernel(const DecodeParams p) {
  griddep_launch_dependents();
  griddep_wait();  // every partial has been written
  const size_t row = blockIdx.x;
  const int d = threadIdx.x;
  const float* ml = p.part_ml + row * p.nchunks * 2;
  const float* po = p.part_o + row * p.nchunks * kHeadDim;
  float M = -INFINITY;
  for (int c = 0; c < p.nchunks; ++c) M = fmaxf(M, ml[2 * c]);
  float l = 0.f, acc = 0.f;
  if (M != -INFINITY) {
    for (int c = 0; c < p.nchunks; ++c) {
      const float w = ex2_approx(ml[2 * c] - M);
      l = fmaf(w, ml[2 * c + 1], l);
      acc = fmaf(w, po[c * kHeadDim + d], acc);
    }
  }
  const float r = l > 0.f ? acc / l : 0.f;
  if (p.out_f32)
    static_cast<float*>(p.out)[row * kHeadDim + d] = r;
  else
    static_cast<__nv_bfloat16*>(p.out)[row * kHeadDim + d] = __float2bfloat16_rn(r);
}

}  // namespace

int decode_chunk_keys() { return kDecChunk; }

// Both kernels use programmatic dependent launch: each may be scheduled
// while the kernel before it in the stream finishes, and waits for it before
// touching global memory.
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.nchunks, p.Lq, p.B * p.H);
  cfg.blockDim = dim3(kDecThreads);
  cfg.stream = stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t e = cudaLaunchKernelEx(&cfg, relpos_decode_partial_kernel, p);
  if (e != cudaSuccess) return e;
  cfg.gridDim = dim3(p.B * p.H * p.Lq);
  cfg.blockDim = dim3(kHeadDim);
  return cudaLaunchKernelEx(&cfg, relpos_decode_combine_kernel, p);
}

}  // namespace relpos

// ---------------------------------------------------------------------------
// Decode without allocation. Some callers cannot allocate device memory at
// call time: code running inside a pre-planned memory budget, or a serving
// loop that must not touch the allocator on the hot path (cudaMallocAsync
// can synchronize or fail when the pool is exhausted). This variant of the
// split-key decode keeps its per-chunk partials in a fixed static device
// array instead of drawing scratch from the stream's pool.

namespace relpos {
namespace {

// Partials of at most kNoAllocScratchBytes: each (query row, key chunk) pair
// needs 66 floats (64 output values, max, sum). Every GPU that loads the
// library holds this array until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

constexpr int kNoAllocMaxDevices = 64;
float* g_noalloc_ptr[kNoAllocMaxDevices];
std::mutex g_noalloc_mu;

// Device address of the static scratch on the current device, looked up once
// per device with that device current (host code cannot use the symbol).
float* noalloc_scratch() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNoAllocMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_noalloc_mu);
  if (!g_noalloc_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess) {
      cudaGetLastError();
      return nullptr;
    }
    g_noalloc_ptr[dev] = static_cast<float*>(ptr);
  }
  return g_noalloc_ptr[dev];
}

// Checks shared by the decode-only entry points, before anything is
// launched: RELPOS_OK to go on, a return code otherwise. *noop is set when
// there is nothing to compute (no query row).
int decode_entry_check(int mode, const void* Q, const void* K, const void* V, const void* bias,
                       const void* key_pos, bool need_key_pos, const void* out, int B, int H,
                       int Lq, int Lk, int num_buckets, int max_distance, int causal,
                       int q_offset, bool* noop) {
  *noop = false;
  int rc = check_rel_params(mode, num_buckets, max_distance, causal);
  if (rc != RELPOS_OK) return rc;
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || q_offset < 0) return RELPOS_ERR_INVALID_ARG;
  if (Lq > 8 && !need_key_pos) return RELPOS_ERR_UNSUPPORTED;  // decode shapes only
  if (B == 0 || H == 0 || Lq == 0) {
    *noop = true;
    return RELPOS_OK;
  }
  if (static_cast<long long>(B) * H > 65535 || Lk > (1 << 24) || q_offset > (1 << 28))
    return RELPOS_ERR_UNSUPPORTED;
  // the kernels read Q, K, V and write out in 16-byte vectors
  if (!Q || !out || !aligned16(Q) || !aligned16(out)) return RELPOS_ERR_INVALID_ARG;
  if (Lk > 0) {
    if (!K || !V || !bias || !aligned16(K) || !aligned16(V)) return RELPOS_ERR_INVALID_ARG;
    if (need_key_pos && (!key_pos || (reinterpret_cast<uintptr_t>(key_pos) & 3u)))
      return RELPOS_ERR_INVALID_ARG;
  }
  return RELPOS_OK;
}

}  // namespace

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

size_t decode_partial_floats(size_t rows, int Lk) {
  const size_t nchunks = (static_cast<size_t>(Lk) + kDecChunk - 1) / kDecChunk;
  return rows * nchunks * (kHeadDim + 2);
}

DecodeParams make_decode_params(const void* Q, const void* K, const void* V, const void* bias,
                                const int* key_pos, int B, int H, int Lq, int Lk, int causal,
                                int q_offset, float scale_log2, const T5Index& t5, int R,
                                float* part, void* out, bool out_f32) {
  DecodeParams dp;
  std::memset(&dp, 0, sizeof(dp));
  dp.Q = static_cast<const __nv_bfloat16*>(Q);
  dp.K = static_cast<const __nv_bfloat16*>(K);
  dp.V = static_cast<const __nv_bfloat16*>(V);
  dp.bias = static_cast<const float*>(bias);
  dp.key_pos = key_pos;
  dp.B = B;
  dp.H = H;
  dp.Lq = Lq;
  dp.Lk = Lk;
  dp.causal = causal;
  dp.q_offset = q_offset;
  dp.scale_log2 = scale_log2;
  dp.chunk = kDecChunk;
  dp.nchunks = (Lk + kDecChunk - 1) / kDecChunk;
  dp.part_o = part;
  dp.part_ml = part + static_cast<size_t>(B) * H * Lq * dp.nchunks * kHeadDim;
  dp.out = out;
  dp.out_f32 = out_f32 ? 1 : 0;
  dp.t5 = t5;
  dp.t5_R = R;
  return dp;
}

}  // namespace relpos

extern "C" int relpos_t5_decode_noalloc(const void* Q, const void* K, const void* V,
                                        const void* bias, int B, int H, int Lq, int Lk,
                                        int num_buckets, int max_distance, int causal,
                                        int q_offset, void* out, void* stream) {
  using namespace relpos;
  bool noop = false;
  int rc = decode_entry_check(RELPOS_T5, Q, K, V, bias, nullptr, false, out, B, H, Lq, Lk, num_buckets,
                              max_distance, causal, q_offset, &noop);
  if (rc != RELPOS_OK || noop) return rc;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t rows = static_cast<size_t>(B) * H * Lq;
  if (Lk == 0)
    return cudaMemsetAsync(out, 0, rows * kHeadDim * 2, s) == cudaSuccess ? RELPOS_OK
                                                                           : RELPOS_ERR_CUDA;
  if (decode_partial_floats(rows, Lk) * sizeof(float) > kNoAllocScratchBytes)
    return RELPOS_ERR_SCRATCH_LIMIT;
  T5Index t5;
  int R = 0;
  const long long nmax = std::max(static_cast<long long>(Lk) - 1,
                                  static_cast<long long>(Lq) - 1 + q_offset);
  rc = t5_setup(num_buckets, max_distance, causal, nmax, &t5, &R);
  if (rc != RELPOS_OK) return rc;
  float* scratch = noalloc_scratch();
  if (!scratch) return RELPOS_ERR_CUDA;
  const float scale_log2 = (1.0f / std::sqrt(static_cast<float>(kHeadDim))) * kLog2e;
  const DecodeParams dp = make_decode_params(Q, K, V, bias, nullptr, B, H, Lq, Lk, causal, q_offset,
                                             scale_log2, t5, R, scratch, out, false);
  if (launch_decode(dp, s) != cudaSuccess) {
    cudaGetLastError();
    return RELPOS_ERR_CUDA;
  }
  return RELPOS_OK;
}

// ---------------------------------------------------------------------------
// Decode over keys at explicit positions: a cache that evicted tokens keeps
// each remaining key at its original position, and an offset-only bias needs
// nothing rewritten ("Relative Position Embeddings, in depth", section
// "Kernels and the KV cache"). Same split-key kernels, with each key's offset
// and causal visibility taken from key_pos.

extern "C" int relpos_t5_decode_positions(const void* Q, const void* K, const void* V,
                                          const void* bias, const int* key_pos, int B, int H,
                                          int Lq, int Lk, int num_buckets, int max_distance,
                                          int causal, int q_offset, void* out, void* stream) {
  using namespace relpos;
  bool noop = false;
  int rc = decode_entry_check(RELPOS_T5, Q, K, V, bias, key_pos, true, out, B, H, Lq, Lk, num_buckets,
                              max_distance, causal, q_offset, &noop);
  if (rc != RELPOS_OK || noop) return rc;
  // more than a few query rows (a chunk of new tokens against the cache): the
  // fused prefill kernel
  if (Lq > 8 && Lk > 0)
    return attn_fwd_t5_positions(Q, K, V, bias, key_pos, B, H, Lq, Lk, num_buckets, max_distance, causal,
                                 q_offset, out, stream);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t rows = static_cast<size_t>(B) * H * Lq;
  if (Lk == 0)
    return cudaMemsetAsync(out, 0, rows * kHeadDim * 2, s) == cudaSuccess ? RELPOS_OK
                                                                           : RELPOS_ERR_CUDA;
  // thresholds for every offset a position in [0, 2^28] can produce
  T5Index t5;
  int R = 0;
  rc = t5_setup(num_buckets, max_distance, causal, (1ll << 28) + 8, &t5, &R);
  if (rc != RELPOS_OK) return rc;
  float* scratch = nullptr;
  if (cudaMallocAsync(&scratch, decode_partial_floats(rows, Lk) * sizeof(float), s) != cudaSuccess) {
    cudaGetLastError();
    return RELPOS_ERR_CUDA;
  }
  const float scale_log2 = (1.0f / std::sqrt(static_cast<float>(kHeadDim))) * kLog2e;
  const DecodeParams dp = make_decode_params(Q, K, V, bias, key_pos, B, H, Lq, Lk, causal, q_offset,
                                             scale_log2, t5, R, scratch, out, false);
  const bool ok = launch_decode(dp, s) == cudaSuccess;
  const bool freed = cudaFreeAsync(scratch, s) == cudaSuccess;
  if (!ok || !freed) {
    cudaGetLastError();
    return RELPOS_ERR_CUDA;
  }
  return RELPOS_OK;
}

// ALiBi over keys at explicit positions: the same split-key kernels with the
// bias -slope_h |key position - query position| ("Relative Position
// Embeddings, in depth", sections "ALiBi and RoPE: the two endpoints" and
// "Kernels and the KV cache"); decode shapes (up to 8 query rows).
extern "C" int relpos_alibi_decode_positions(const void* Q, const void* K, const void* V,
                                             const void* slopes, const int* key_pos, int B, int H,
                                             int Lq, int Lk, int causal, int q_offset, void* out,
                                             void* stream) {
  using namespace relpos;
  bool noop = false;
  int rc = decode_entry_check(RELPOS_ALIBI, Q, K, V, slopes, key_pos, true, out, B, H, Lq, Lk, 0, 0, causal,
                              q_offset, &noop);
  if (rc != RELPOS_OK || noop) return rc;
  if (Lq > 8) return RELPOS_ERR_UNSUPPORTED;
  if (Lk > 0 && (reinterpret_cast<uintptr_t>(slopes) & 3u)) return RELPOS_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t rows = static_cast<size_t>(B) * H * Lq;
  if (Lk == 0)
    return cudaMemsetAsync(out, 0, rows * kHeadDim * 2, s) == cudaSuccess ? RELPOS_OK
                                                                           : RELPOS_ERR_CUDA;
  float* scratch = nullptr;
  if (cudaMallocAsync(&scratch, decode_partial_floats(rows, Lk) * sizeof(float), s) != cudaSuccess) {
    cudaGetLastError();
    return RELPOS_ERR_CUDA;
  }
  T5Index unused;
  std::memset(&unused, 0, sizeof(unused));
  const float scale_log2 = (1.0f / std::sqrt(static_cast<float>(kHeadDim))) * kLog2e;
  // t5_R = -1 selects the ALiBi bias in the partial kernel
  const DecodeParams dp = make_decode_params(Q, K, V, slopes, key_pos, B, H, Lq, Lk, causal, q_offset,
                                             scale_log2, unused, -1, scratch, out, false);
  const bool ok = launch_decode(dp, s) == cudaSuccess;
  const bool freed = cudaFreeAsync(scratch, s) == cudaSuccess;
  if (!ok || !freed) {
    cudaGetLastError();
    return RELPOS_ERR_CUDA;
  }
  return RELPOS_OK;
}
