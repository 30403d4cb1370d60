// api.cu -- the C ABI (include/relpos_attn.h): argument checks, the T5
// bucket thresholds, TMA descriptors, scratch management and dispatch to the
// fused prefill kernel or the split-key decode kernel.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <climits>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "../../include/relpos_attn.h"
#include "ptx.cuh"
#include "relpos_bwd.cuh"
#include "relpos_common.cuh"
#include "relpos_internal.h"

namespace relpos {
namespace {

// Device status word: kernels record the first bounded-wait failure here.
__device__ int g_status;

constexpr int kMaxDevices = 64;
int* g_status_ptr[kMaxDevices];
std::mutex g_status_mu;

int* status_ptr() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_status_mu);
  if (!g_status_ptr[dev]) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_status) != cudaSuccess) return nullptr;
    g_status_ptr[dev] = static_cast<int*>(ptr);
  }
  return g_status_ptr[dev];
}

int g_num_sms[kMaxDevices];

int num_sms() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return -1;
  if (g_num_sms[dev] <= 0) {
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return -1;
    g_num_sms[dev] = n;
  }
  return g_num_sms[dev];
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<PFN_cuTensorMapEncodeTiled_v12000>(nullptr);
    return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }();
  return fn;
}

// [rows = L, inner = 64] bf16 per (batch*head) slab, 128-row x 64-col boxes,
// 128-byte swizzle (the operand layout of the tensor-core descriptors).
// `inner` columns per row (64, or 128 for Transformer-XL's query rows, read
// as two 64-column boxes).
bool make_tmap(CUtensorMap* m, const void* base, int L, int BH, int inner = kHeadDim) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(inner) * 2,
                           static_cast<cuuint64_t>(L) * inner * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), 128u, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// DeBERTa table [rows = 2k, H, 64] bf16: boxes of 64 table rows of one head
bool make_tmap_table(CUtensorMap* m, const void* base, int H, int rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(H),
                        static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 2,
                           static_cast<cuuint64_t>(H) * kHeadDim * 2};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(kHeadDim), 1u, 64u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// fp32 [rows = L, inner = 64] per (batch*head) slab, 128-row x 32-column
// boxes, 128-byte swizzle (the backward's dQ accumulator)
bool make_tmap_acc(CUtensorMap* m, const void* base, int L, int BH) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(kHeadDim), static_cast<cuuint64_t>(L),
                        static_cast<cuuint64_t>(BH)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(kHeadDim) * 4,
                           static_cast<cuuint64_t>(L) * kHeadDim * 4};
  cuuint32_t box[3] = {32u, 128u, 1u};
  cuuint32_t estr[3] = {1u, 1u, 1u};
  CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<void*>(base), dims, strides, box, estr,
                  CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

}  // namespace

// Thresholds of the T5 log buckets: thr[q] is the smallest distance n whose
// bucket within a half is >= exact + q + 1, found by evaluating the pages'
// formula exact + int(log(n / exact) / log(max_distance / exact) * (S - exact))
// in double precision for n = exact, exact + 1, ... up to saturation or nmax.
// R is the first distance of the last bucket (nmax + 1 if not reached).
int t5_setup(int num_buckets, int max_distance, int causal, long long nmax, T5Index* ix, int* R) {
  std::memset(ix, 0, sizeof(*ix));
  ix->bidir = causal ? 0 : 1;
  ix->slots = causal ? num_buckets : num_buckets / 2;
  ix->exact = ix->slots / 2;
  ix->nthr = ix->slots - ix->exact - 1;
  for (int q = 0; q < kMaxT5Thresholds; ++q) ix->thr[q] = INT_MAX;
  if (ix->nthr == 0) {
    *R = ix->exact;
    return RELPOS_OK;
  }
  const int S = ix->slots, E = ix->exact;
  const double denom = std::log(static_cast<double>(max_distance) / static_cast<double>(E));
  int cur = E;
  for (long long n = E; n <= nmax && cur < S - 1; ++n) {
    const double v = std::log(static_cast<double>(n) / static_cast<double>(E)) / denom *
                     static_cast<double>(S - E);
    long long large = E + static_cast<long long>(v);
    if (large > S - 1) large = S - 1;
    if (large < cur) return RELPOS_ERR_UNSUPPORTED;  // log not monotone here
    while (cur < large) {
      ++cur;
      ix->thr[cur - E - 1] = static_cast<int>(n);
    }
  }
  *R = (cur == S - 1) ? ix->thr[ix->nthr - 1] : static_cast<int>(nmax + 1);
  return RELPOS_OK;
}

int check_rel_params(int mode, int num_buckets, int rel_param, int causal) {
  if (causal != 0 && causal != 1) return RELPOS_ERR_INVALID_ARG;
  if (mode == RELPOS_T5) {
    if (num_buckets < 4 || num_buckets > 128 || (num_buckets & 1)) return RELPOS_ERR_INVALID_ARG;
    const int S = causal ? num_buckets : num_buckets / 2;
    if (rel_param <= S / 2) return RELPOS_ERR_INVALID_ARG;  // log(max_distance / exact) <= 0
  } else if (mode == RELPOS_SHAW || mode == RELPOS_DEBERTA) {
    if (rel_param < 1) return RELPOS_ERR_INVALID_ARG;
    if (rel_param > (1 << 24)) return RELPOS_ERR_UNSUPPORTED;
  } else if (mode != RELPOS_ALIBI && mode != RELPOS_TXL) {
    return RELPOS_ERR_INVALID_ARG;
  }
  return RELPOS_OK;
}

namespace {

__global__ void index_ids_kernel(int mode, int n, int first, T5Index ix, int k, int* out) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= n) return;
  const int rel = first + i;
  int id;
  if (mode == RELPOS_T5)
    id = t5_bucket_dev(rel, ix);
  else if (mode == RELPOS_SHAW)
    id = shaw_index_dev(rel, k);
  else if (mode == RELPOS_ALIBI)
    id = rel < 0 ? -rel : rel;
  else if (mode == RELPOS_TXL)
    id = -rel;
  else
    id = deberta_delta_dev(rel, k);
  out[i] = id;
}

__global__ void selftest_wait_kernel(unsigned long long limit_ns, int* status) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nothing ever arrives: phase 0 cannot complete
    if (!mbar_wait(smem_u32(&bar), 0, limit_ns)) atomicCAS(status, 0, RELPOS_ERR_DEVICE_TIMEOUT);
  }
}

__global__ void f32_to_bf16_kernel(const float4* __restrict__ in, uint2* __restrict__ out, size_t n4) {
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < n4;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    const float4 v = in[i];
    uint2 o;
    o.x = pack_bf16x2(v.x, v.y);
    o.y = pack_bf16x2(v.z, v.w);
    out[i] = o;
  }
}

cudaError_t to_bf16(const void* src, void* dst, size_t n, cudaStream_t s) {
  const size_t n4 = n / 4;  // n is a multiple of 64
  int blocks = static_cast<int>((n4 + 255) / 256);
  if (blocks > 152 * 16) blocks = 152 * 16;
  if (blocks < 1) blocks = 1;
  f32_to_bf16_kernel<<<blocks, 256, 0, s>>>(static_cast<const float4*>(src), static_cast<uint2*>(dst),
                                             n4);
  return cudaGetLastError();
}

}  // namespace
}  // namespace relpos

using namespace relpos;

extern "C" const char* relpos_strerror(int code) {
  switch (code) {
    case RELPOS_OK: return "ok";
    case RELPOS_ERR_INVALID_ARG: return "invalid argument";
    case RELPOS_ERR_UNSUPPORTED: return "unsupported by this build";
    case RELPOS_ERR_CUDA: return "CUDA error";
    case RELPOS_ERR_DEVICE_TIMEOUT: return "device-side bounded wait timed out";
    case RELPOS_ERR_SCRATCH_LIMIT: return "request exceeds the fixed scratch of the no-allocation decode";
    default: return "unknown error";
  }
}

extern "C" int relpos_index_ids(int mode, int n, int rel_first, int num_buckets, int rel_param,
                                int causal, int* out_dev, void* stream) {
  int rc = check_rel_params(mode, num_buckets, rel_param, causal);
  if (rc != RELPOS_OK) return rc;
  if (n < 0) return RELPOS_ERR_INVALID_ARG;
  if (n == 0) return RELPOS_OK;
  if (!out_dev) return RELPOS_ERR_INVALID_ARG;
  const long long last = static_cast<long long>(rel_first) + n - 1;
  if (rel_first < -(1 << 30) || last > (1 << 30)) return RELPOS_ERR_UNSUPPORTED;
  T5Index ix;
  std::memset(&ix, 0, sizeof(ix));
  if (mode == RELPOS_T5) {
    int R = 0;
    const long long nmax = std::max(std::llabs(static_cast<long long>(rel_first)), std::llabs(last));
    rc = t5_setup(num_buckets, rel_param, causal, nmax, &ix, &R);
    if (rc != RELPOS_OK) return rc;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  index_ids_kernel<<<(n + 255) / 256, 256, 0, s>>>(mode, n, rel_first, ix, rel_param, out_dev);
  return cudaGetLastError() == cudaSuccess ? RELPOS_OK : RELPOS_ERR_CUDA;
}

extern "C" int relpos_check_status(void* stream) {
  if (cudaStreamSynchronize(static_cast<cudaStream_t>(stream)) != cudaSuccess) {
    cudaGetLastError();
    return RELPOS_ERR_CUDA;
  }
  int* sp = status_ptr();
  if (!sp) return RELPOS_ERR_CUDA;
  int v = 0;
  if (cudaMemcpy(&v, sp, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return RELPOS_ERR_CUDA;
  if (v != 0) {
    const int zero = 0;
    if (cudaMemcpy(sp, &zero, sizeof(int), cudaMemcpyHostToDevice) != cudaSuccess)
      return RELPOS_ERR_CUDA;
    return RELPOS_ERR_DEVICE_TIMEOUT;
  }
  return RELPOS_OK;
}

extern "C" int relpos_selftest_wait_timeout(int timeout_us, void* stream) {
  if (timeout_us < 1 || timeout_us > 1000000) return RELPOS_ERR_INVALID_ARG;
  int* sp = status_ptr();
  if (!sp) return RELPOS_ERR_CUDA;
  selftest_wait_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<unsigned long long>(timeout_us) * 1000ull, sp);
  return cudaGetLastError() == cudaSuccess ? RELPOS_OK : RELPOS_ERR_CUDA;
}

namespace relpos {
namespace {

// relpos_attn_fwd and relpos_attn_fwd_padded; lengths (device int32 [B]) is
// null for an unpadded batch. key_pos (device int32 [B, H, Lk], T5 only) puts
// every key at an explicit position; null for keys at their index.
int attn_fwd_impl(int mode, int dtype, const void* Q, const void* K, const void* V,
                  const void* table0, const void* table1, const int* lengths, const int* key_pos, int B,
                  int H, int Lq, int Lk, int d, int num_buckets, int rel_param, int causal, int q_offset,
                  void* out, void* stream) {
  if (mode != RELPOS_T5 && mode != RELPOS_SHAW && mode != RELPOS_DEBERTA && mode != RELPOS_ALIBI &&
      mode != RELPOS_TXL)
    return RELPOS_ERR_INVALID_ARG;
  if (dtype != RELPOS_BF16 && dtype != RELPOS_FP32) return RELPOS_ERR_INVALID_ARG;
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || q_offset < 0 || d <= 0) return RELPOS_ERR_INVALID_ARG;
  int rc = check_rel_params(mode, num_buckets, rel_param, causal);
  if (rc != RELPOS_OK) return rc;
  if (key_pos && (mode != RELPOS_T5 || dtype != RELPOS_BF16 || d != kHeadDim || lengths))
    return RELPOS_ERR_UNSUPPORTED;
  // d = 64 throughout; d = 128 for T5 and ALiBi with bf16 inputs
  if (d != kHeadDim &&
      !(d == 2 * kHeadDim && (mode == RELPOS_T5 || mode == RELPOS_ALIBI) && dtype == RELPOS_BF16))
    return RELPOS_ERR_UNSUPPORTED;
  if (B == 0 || H == 0 || Lq == 0) return RELPOS_OK;
  if (!Q || !out) return RELPOS_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > 65535) return RELPOS_ERR_UNSUPPORTED;
  if (Lq > (1 << 24) || Lk > (1 << 24) || q_offset > (1 << 28)) return RELPOS_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t esz = dtype == RELPOS_FP32 ? 4 : 2;
  const size_t BH = static_cast<size_t>(B) * H;
  if (Lk == 0) {  // no key is visible: zero rows
    return cudaMemsetAsync(out, 0, BH * Lq * static_cast<size_t>(d) * esz, s) == cudaSuccess
               ? RELPOS_OK
               : RELPOS_ERR_CUDA;
  }
  if (!K || !V || !table0) return RELPOS_ERR_INVALID_ARG;
  if ((mode == RELPOS_SHAW || mode == RELPOS_DEBERTA || mode == RELPOS_TXL) && !table1)
    return RELPOS_ERR_INVALID_ARG;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || !aligned16(out) || !aligned16(table0) ||
      (table1 && !aligned16(table1)))
    return RELPOS_ERR_INVALID_ARG;
  if (mode == RELPOS_DEBERTA && rel_param > 4096) return RELPOS_ERR_UNSUPPORTED;
  // Shaw's 2k + 1 table rows are one 64-row tensor-core operand
  if (mode == RELPOS_SHAW && 2 * rel_param + 1 > 64) return RELPOS_ERR_UNSUPPORTED;

  int* status = status_ptr();
  if (!status) return RELPOS_ERR_CUDA;

  // relative-term setup
  T5Index t5;
  std::memset(&t5, 0, sizeof(t5));
  int R = 0;
  if (mode == RELPOS_T5) {
    // explicit positions: thresholds for every offset a position in [0, 2^28] can produce
    const long long nmax = key_pos ? (1ll << 28) + Lq + static_cast<long long>(q_offset)
                                   : std::max(static_cast<long long>(Lk) - 1,
                                              static_cast<long long>(Lq) - 1 + q_offset);
    rc = t5_setup(num_buckets, rel_param, causal, nmax, &t5, &R);
    if (rc != RELPOS_OK) return rc;
  }
  const float scale = 1.0f / std::sqrt(static_cast<float>(mode == RELPOS_DEBERTA ? 3 * d : d));

  // fp32 inputs: round to bf16 scratch first
  void* scratch = nullptr;
  const void* Qb = Q;
  const void* Kb = K;
  const void* Vb = V;
  const size_t nq = BH * Lq * d, nk = BH * Lk * d;
  auto fail = [&](int code) {
    if (scratch) cudaFreeAsync(scratch, s);
    cudaGetLastError();
    return code;
  };
  const bool decode = (mode == RELPOS_T5 && Lq <= 8 && !lengths && !key_pos && d == kHeadDim);
  size_t scratch_bytes = 0, off_conv = 0, off_part = 0;
  if (dtype == RELPOS_FP32) {
    off_conv = scratch_bytes;
    scratch_bytes += (nq + 2 * nk) * 2;
  }
  if (decode) {
    scratch_bytes = (scratch_bytes + 255) & ~static_cast<size_t>(255);
    off_part = scratch_bytes;
    scratch_bytes += decode_partial_floats(BH * Lq, Lk) * sizeof(float);
  }
  // DeBERTa: the band array [BH, Lq, band_pitch] (bf16, with kBandPad bytes
  // before and after it: the attention kernel reads whole 128-key windows
  // that may start up to 254 columns before a row and end up to 261 after
  // the band, the part outside being replaced by the far terms), C2P's two
  // saturated columns per query row and P2C's per key (fp32)
  const size_t n2k = 2 * static_cast<size_t>(rel_param);
  const int band_pitch = static_cast<int>((n2k + 8 + 7) & ~static_cast<size_t>(7));
  const int const_pitch = (Lq + 127) & ~127;
  const int ends_pitch = (Lk + 127) & ~127;
  constexpr size_t kBandPad = 1024;
  size_t off_band = 0, off_const = 0, off_ends = 0;
  if (mode == RELPOS_DEBERTA) {
    scratch_bytes = (scratch_bytes + 255) & ~static_cast<size_t>(255);
    off_band = scratch_bytes + kBandPad;
    scratch_bytes += ((BH * Lq * band_pitch * 2 + 2 * kBandPad) + 255) & ~static_cast<size_t>(255);
    off_const = scratch_bytes;
    scratch_bytes += BH * 2 * static_cast<size_t>(const_pitch) * sizeof(float);
    off_ends = scratch_bytes;
    scratch_bytes += BH * 2 * static_cast<size_t>(ends_pitch) * sizeof(float);
  }
  // Transformer-XL: the 128-wide query rows [BH, Lq, 128] and the keys'
  // sinusoid table [Lk, 64] (bf16)
  size_t off_q2 = 0, off_sin = 0;
  if (mode == RELPOS_TXL) {
    scratch_bytes = (scratch_bytes + 255) & ~static_cast<size_t>(255);
    off_q2 = scratch_bytes;
    scratch_bytes += BH * Lq * 2 * kHeadDim * 2;
    scratch_bytes = (scratch_bytes + 255) & ~static_cast<size_t>(255);
    off_sin = scratch_bytes;
    scratch_bytes += static_cast<size_t>(Lk) * kHeadDim * 2;
  }
  if (scratch_bytes) {
    if (cudaMallocAsync(&scratch, scratch_bytes, s) != cudaSuccess) return fail(RELPOS_ERR_CUDA);
  }
  if (dtype == RELPOS_FP32) {
    uint8_t* c = static_cast<uint8_t*>(scratch) + off_conv;
    if (to_bf16(Q, c, nq, s) != cudaSuccess || to_bf16(K, c + nq * 2, nk, s) != cudaSuccess ||
        to_bf16(V, c + (nq + nk) * 2, nk, s) != cudaSuccess)
      return fail(RELPOS_ERR_CUDA);
    Qb = c;
    Kb = c + nq * 2;
    Vb = c + (nq + nk) * 2;
  }

  if (decode) {
    float* part = reinterpret_cast<float*>(static_cast<uint8_t*>(scratch) + off_part);
    const DecodeParams dp = make_decode_params(Qb, Kb, Vb, table0, nullptr, B, H, Lq, Lk, causal,
                                               q_offset, scale * kLog2e, t5, R, part, out,
                                               dtype == RELPOS_FP32);
    if (launch_decode(dp, s) != cudaSuccess) return fail(RELPOS_ERR_CUDA);
  } else {
    FwdParams p;
    std::memset(&p, 0, sizeof(p));
    p.B = B;
    p.H = H;
    p.Lq = Lq;
    p.Lk = Lk;
    p.dh = d;
    p.causal = causal;
    p.q_offset = q_offset;
    p.scale_log2 = scale * kLog2e;
    p.out = out;
    p.out_v8 = (reinterpret_cast<uintptr_t>(out) & 31u) == 0;
    // long items of mostly far tiles: causal T5 and Transformer-XL
    p.stagger = (mode == RELPOS_T5 || mode == RELPOS_TXL) && causal;
    p.status = status;
    p.kclip = rel_param;
    p.Qg = static_cast<const __nv_bfloat16*>(Qb);
    p.npairs = (Lq + 255) / 256;
    p.lengths = lengths;
    p.key_pos = key_pos;
    if (key_pos) p.stagger = 0;
    // split items balance a last pass of equally long items: not with padding
    // or explicit positions
    p.nsplit = (lengths || key_pos) ? 0 : fwd_split_items(B * H * p.npairs, B * H, Lq, causal, num_sms());
    if (mode == RELPOS_T5) {
      p.bias = static_cast<const float*>(table0);
      p.t5 = t5;
      p.t5_R = R;
      p.t5_nb = num_buckets;
      p.t5_tab_off = R + 254;
      p.t5_tab_len = 2 * R + 509;
      p.t5_tab_len4 = (p.t5_tab_len + 3) & ~3;
    } else if (mode == RELPOS_SHAW) {
      p.aK = static_cast<const __nv_bfloat16*>(table0);
      p.aV = static_cast<const __nv_bfloat16*>(table1);
    } else if (mode == RELPOS_ALIBI) {
      p.slopes = static_cast<const float*>(table0);
    }
    // Shaw per-row tables: padded rows when shared memory allows
    p.row_stride = 2 * rel_param + 2;
    if (mode == RELPOS_SHAW && fwd_smem_bytes(mode, p) > fwd_max_smem_bytes()) p.row_stride = 2 * rel_param + 1;
    // T5: one table copy when the four shifted copies do not fit
    if (mode == RELPOS_T5 && fwd_smem_bytes(mode, p) > fwd_max_smem_bytes()) p.t5_compact = 1;
    if (p.nsplit > 0 && fwd_smem_bytes(mode, p) > fwd_max_smem_bytes()) p.nsplit = 0;
    if (fwd_smem_bytes(mode, p) > fwd_max_smem_bytes()) return fail(RELPOS_ERR_UNSUPPORTED);
    if (mode == RELPOS_DEBERTA) {
      uint8_t* sc = static_cast<uint8_t*>(scratch);
      BandParams bp;
      std::memset(&bp, 0, sizeof(bp));
      bp.BH = static_cast<int>(BH);
      bp.H = H;
      bp.k = rel_param;
      bp.Lq = Lq;
      bp.Lk = Lk;
      bp.q_offset = q_offset;
      bp.scale = scale * kLog2e;
      bp.K = static_cast<const __nv_bfloat16*>(Kb);
      bp.Pq = static_cast<const __nv_bfloat16*>(table1);
      bp.band = reinterpret_cast<__nv_bfloat16*>(sc + off_band);
      bp.band_pitch = band_pitch;
      bp.c2p_const = reinterpret_cast<float*>(sc + off_const);
      bp.const_pitch = const_pitch;
      bp.ends = reinterpret_cast<float*>(sc + off_ends);
      bp.ends_pitch = ends_pitch;
      bp.status = status;
      p.band = bp.band;
      p.band_pitch = band_pitch;
      p.c2p_const = bp.c2p_const;
      p.const_pitch = const_pitch;
      p.p2c_ends = bp.ends;
      p.ends_pitch = ends_pitch;
      CUtensorMap tqa, tka, tpk, tpq;
      if (!make_tmap_table(&tpk, table0, H, static_cast<int>(n2k)) ||
          !make_tmap_table(&tpq, table1, H, static_cast<int>(n2k)) ||
          !make_tmap(&tqa, Qb, Lq, static_cast<int>(BH)) || !make_tmap(&tka, Kb, Lk, static_cast<int>(BH)))
        return fail(RELPOS_ERR_CUDA);
      if (launch_deberta_band(tqa, tka, tpk, tpq, bp, s) != cudaSuccess) return fail(RELPOS_ERR_CUDA);
    }
    CUtensorMap tq, tk, tv, ts;
    if (mode == RELPOS_TXL) {
      uint8_t* sc = static_cast<uint8_t*>(scratch);
      TxlParams tp;
      std::memset(&tp, 0, sizeof(tp));
      tp.BH = static_cast<int>(BH);
      tp.H = H;
      tp.Lq = Lq;
      tp.Lk = Lk;
      tp.q_offset = q_offset;
      tp.Q = static_cast<const __nv_bfloat16*>(Qb);
      tp.W = static_cast<const float*>(table0);
      tp.uv = static_cast<const float*>(table1);
      tp.Q2 = reinterpret_cast<__nv_bfloat16*>(sc + off_q2);
      tp.Ksin = reinterpret_cast<__nv_bfloat16*>(sc + off_sin);
      tp.status = status;
      for (int m = 0; m < kHeadDim / 2; ++m)
        tp.omega[m] = static_cast<float>(std::pow(10000.0, -2.0 * m / kHeadDim));
      if (launch_txl_prep(tp, s) != cudaSuccess) return fail(RELPOS_ERR_CUDA);
      if (!make_tmap(&tq, tp.Q2, Lq, static_cast<int>(BH), 2 * kHeadDim) ||
          !make_tmap(&ts, tp.Ksin, Lk, 1))
        return fail(RELPOS_ERR_CUDA);
    } else if (!make_tmap(&tq, Qb, Lq, static_cast<int>(BH), d)) {
      return fail(RELPOS_ERR_CUDA);
    }
    if (!make_tmap(&tk, Kb, Lk, static_cast<int>(BH), d) || !make_tmap(&tv, Vb, Lk, static_cast<int>(BH), d))
      return fail(RELPOS_ERR_CUDA);
    if (mode != RELPOS_TXL) ts = tk;  // unused
    const int sms = num_sms();
    if (sms <= 0) return fail(RELPOS_ERR_CUDA);
    if (launch_fwd(mode, dtype == RELPOS_FP32, tq, tk, tv, ts, p, sms, s) != cudaSuccess)
      return fail(RELPOS_ERR_CUDA);
  }
  if (scratch && cudaFreeAsync(scratch, s) != cudaSuccess) {
    cudaGetLastError();
    return RELPOS_ERR_CUDA;
  }
  return RELPOS_OK;
}

}  // namespace
}  // namespace relpos

extern "C" int relpos_attn_fwd(int mode, int dtype, const void* Q, const void* K, const void* V,
                               const void* table0, const void* table1, int B, int H, int Lq, int Lk,
                               int d, int num_buckets, int rel_param, int causal, int q_offset,
                               void* out, void* stream) {
  return attn_fwd_impl(mode, dtype, Q, K, V, table0, table1, nullptr, nullptr, B, H, Lq, Lk, d,
                       num_buckets, rel_param, causal, q_offset, out, stream);
}

extern "C" int relpos_attn_fwd_padded(int mode, int dtype, const void* Q, const void* K,
                                      const void* V, const void* table0, const void* table1,
                                      const int* lengths, int B, int H, int Lq, int Lk, int d,
                                      int num_buckets, int rel_param, int causal, int q_offset,
                                      void* out, void* stream) {
  if (!lengths || (reinterpret_cast<uintptr_t>(lengths) & 3u)) return RELPOS_ERR_INVALID_ARG;
  return attn_fwd_impl(mode, dtype, Q, K, V, table0, table1, lengths, nullptr, B, H, Lq, Lk, d,
                       num_buckets, rel_param, causal, q_offset, out, stream);
}

namespace relpos {
int attn_fwd_t5_positions(const void* Q, const void* K, const void* V, const void* bias, const int* key_pos,
                          int B, int H, int Lq, int Lk, int num_buckets, int max_distance, int causal,
                          int q_offset, void* out, void* stream) {
  return attn_fwd_impl(RELPOS_T5, RELPOS_BF16, Q, K, V, bias, nullptr, nullptr, key_pos, B, H, Lq, Lk,
                       kHeadDim, num_buckets, max_distance, causal, q_offset, out, stream);
}
}  // namespace relpos

namespace relpos {
namespace {

// relpos_t5_attn_bwd (mode 0: table = bias [nb, H], dtable = dbias),
// relpos_shaw_attn_bwd (mode 1: table / table1 = a_K / a_V [2k + 1, 64] bf16,
// dtable / dtable1 = their fp32 gradients, max_distance = k),
// relpos_deberta_attn_bwd (mode 2: table / table1 = Pk / Pq [2k, H, 64] bf16,
// dtable / dtable1 = their fp32 gradients, max_distance = k) and
// relpos_alibi_attn_bwd (mode 3: table = slopes [H], dtable = dslopes).
int attn_bwd_impl(int mode, const void* Q, const void* K, const void* V, const void* dO,
                  const void* table, const void* table1, int B, int H, int Lq, int Lk, int d, int num_buckets,
                  int max_distance, int causal, int q_offset, void* dQ, void* dK, void* dV,
                  void* dtable, void* dtable1, void* stream) {
  if (B < 0 || H < 0 || Lq < 0 || Lk < 0 || q_offset < 0 || d <= 0) return RELPOS_ERR_INVALID_ARG;
  int rc = check_rel_params(mode, num_buckets, max_distance, causal);
  if (rc != RELPOS_OK) return rc;
  if (d != kHeadDim) return RELPOS_ERR_UNSUPPORTED;
  if (mode == RELPOS_SHAW && max_distance > bwd_max_shaw_k()) return RELPOS_ERR_UNSUPPORTED;
  if (mode == RELPOS_DEBERTA && max_distance > 4096) return RELPOS_ERR_UNSUPPORTED;
  if (B == 0 || H == 0) return RELPOS_OK;
  if (!table || !dtable || !aligned16(table) || !aligned16(dtable)) return RELPOS_ERR_INVALID_ARG;
  if ((mode == RELPOS_SHAW || mode == RELPOS_DEBERTA) &&
      (!table1 || !dtable1 || !aligned16(table1) || !aligned16(dtable1)))
    return RELPOS_ERR_INVALID_ARG;
  if (static_cast<long long>(B) * H > 65535) return RELPOS_ERR_UNSUPPORTED;
  if (Lq > (1 << 24) || Lk > (1 << 24) || q_offset > (1 << 28)) return RELPOS_ERR_UNSUPPORTED;
  // every pointer is checked before anything (the table gradient's clear
  // included) is queued
  if (Lq > 0 && (!dQ || !aligned16(dQ))) return RELPOS_ERR_INVALID_ARG;
  if (Lk > 0 && (!dK || !dV || !aligned16(dK) || !aligned16(dV))) return RELPOS_ERR_INVALID_ARG;
  if (Lq > 0 && Lk > 0) {
    for (const void* ptr : {Q, K, V, dO})
      if (!ptr || !aligned16(ptr)) return RELPOS_ERR_INVALID_ARG;
  }
  T5Index t5;
  std::memset(&t5, 0, sizeof(t5));
  int R = 0;
  if (mode == RELPOS_T5) {
    const long long nmax =
        std::max(static_cast<long long>(Lk) - 1, static_cast<long long>(Lq) - 1 + q_offset);
    rc = t5_setup(num_buckets, max_distance, causal, nmax, &t5, &R);
    if (rc != RELPOS_OK) return rc;
    if (Lq > 0 && Lk > 0 && (R < 1 || R > bwd_max_R())) return RELPOS_ERR_UNSUPPORTED;
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t BH = static_cast<size_t>(B) * H;
  const size_t row_bytes = kHeadDim * 2;
  const size_t dtable_bytes =
      (mode == RELPOS_T5        ? static_cast<size_t>(num_buckets) * H
       : mode == RELPOS_SHAW    ? static_cast<size_t>(2 * max_distance + 1) * kHeadDim
       : mode == RELPOS_DEBERTA ? static_cast<size_t>(2 * max_distance) * H * kHeadDim
                                : static_cast<size_t>(H)) *
      sizeof(float);
  if (cudaMemsetAsync(dtable, 0, dtable_bytes, s) != cudaSuccess) return RELPOS_ERR_CUDA;
  if ((mode == RELPOS_SHAW || mode == RELPOS_DEBERTA) && cudaMemsetAsync(dtable1, 0, dtable_bytes, s) != cudaSuccess)
    return RELPOS_ERR_CUDA;
  if (Lq == 0 || Lk == 0) {  // no score: every gradient is zero
    bool ok = true;
    if (Lq > 0) ok = ok && cudaMemsetAsync(dQ, 0, BH * Lq * row_bytes, s) == cudaSuccess;
    if (Lk > 0) ok = ok && cudaMemsetAsync(dK, 0, BH * Lk * row_bytes, s) == cudaSuccess &&
                      cudaMemsetAsync(dV, 0, BH * Lk * row_bytes, s) == cudaSuccess;
    return ok ? RELPOS_OK : RELPOS_ERR_CUDA;
  }
  int* status = status_ptr();
  if (!status) return RELPOS_ERR_CUDA;

  // scratch: the fp32 dQ accumulator, then the row statistics (lse, D) with
  // rows padded to whole 128-row query tiles; Shaw: the rows' end values,
  // their T, U and per-offset sums of P and dS (2k + 2 floats a row), and
  // every query tile's partial table gradients
  const int lq_pad = (Lq + 127) & ~127;
  const size_t n_acc = BH * Lq * kHeadDim, n_stats = 2 * BH * static_cast<size_t>(lq_pad);
  const int nr = mode == RELPOS_SHAW ? 2 * max_distance + 2 : 0;
  const size_t n_rows = BH * static_cast<size_t>(lq_pad);
  const size_t n_shaw = mode == RELPOS_SHAW ? 4 * n_rows + 4 * n_rows * nr +
                                                  n_rows / 128 * 2 * static_cast<size_t>(2 * max_distance + 1) * kHeadDim
                                            : 0;
  // DeBERTa (in floats, each part a multiple of 64): the band pre-pass arrays
  // (bf16 band rows with a pad on each side, the rows' saturated c2p values,
  // the keys' saturated p2c values), dS gathered by table row query- and
  // key-major (bf16), the rows' and keys' dS beyond the band, the fp32 dK
  const int lk_pad = (Lk + 127) & ~127;
  const size_t k2 = 2 * static_cast<size_t>(max_distance);
  const int band_pitch = static_cast<int>((k2 + 8 + 7) & ~static_cast<size_t>(7));
  auto r64 = [](size_t n) { return (n + 63) & ~static_cast<size_t>(63); };
  size_t n_deb = 0, o_band = 0, o_c2p = 0, o_ends = 0, o_dsq = 0, o_dsk = 0, o_rowfar = 0, o_keyfar = 0, o_dk = 0,
         o_m1 = 0, o_mk = 0, o_e4 = 0;
  if (mode == RELPOS_DEBERTA) {
    const size_t base = n_acc + n_stats;
    o_band = base + 256;  // 1 KB before the band rows
    n_deb = r64(256 + (BH * Lq * band_pitch + 1) / 2 + 256);
    o_c2p = base + n_deb;
    n_deb += r64(BH * 2 * lq_pad);
    o_ends = base + n_deb;
    n_deb += r64(BH * 2 * lk_pad);
    o_dsq = base + n_deb;
    n_deb += r64(BH * lq_pad * k2 / 2);
    o_dsk = base + n_deb;
    n_deb += r64(BH * lk_pad * k2 / 2);
    o_rowfar = base + n_deb;
    n_deb += r64(BH * 2 * lq_pad);
    o_keyfar = base + n_deb;
    n_deb += r64(2 * BH * 2 * lk_pad);
    o_dk = base + n_deb;
    n_deb += r64(BH * Lk * kHeadDim);
    o_m1 = base + n_deb;  // then the fp32 band members of the saturated rows
    n_deb += r64(BH * lq_pad);
    o_mk = base + n_deb;
    n_deb += r64(BH * lk_pad);
    o_e4 = base + n_deb;  // the rows' values for the sub-steps beyond the band
    n_deb += r64(BH * 4 * lq_pad);
  }
  float* scratch = nullptr;
  if (cudaMallocAsync(reinterpret_cast<void**>(&scratch), (n_acc + n_stats + n_shaw + n_deb) * sizeof(float), s) !=
      cudaSuccess) {
    cudaGetLastError();
    return RELPOS_ERR_CUDA;
  }
  auto done = [&](int code) {
    if (cudaFreeAsync(scratch, s) != cudaSuccess && code == RELPOS_OK) code = RELPOS_ERR_CUDA;
    if (code != RELPOS_OK) cudaGetLastError();
    return code;
  };
  if (cudaMemsetAsync(scratch, 0, n_acc * sizeof(float), s) != cudaSuccess) return done(RELPOS_ERR_CUDA);
  CUtensorMap tq, tk, tv, tdo, tacc;
  if (!make_tmap(&tq, Q, Lq, static_cast<int>(BH)) || !make_tmap(&tk, K, Lk, static_cast<int>(BH)) ||
      !make_tmap(&tv, V, Lk, static_cast<int>(BH)) || !make_tmap(&tdo, dO, Lq, static_cast<int>(BH)) ||
      !make_tmap_acc(&tacc, scratch, Lq, static_cast<int>(BH)))
    return done(RELPOS_ERR_CUDA);
  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  p.B = B;
  p.H = H;
  p.Lq = Lq;
  p.Lk = Lk;
  p.causal = causal;
  p.q_offset = q_offset;
  p.scale = 1.0f / std::sqrt(static_cast<float>(d));
  p.scale_log2 = p.scale * kLog2e;
  if (mode == RELPOS_T5) {
    p.bias = static_cast<const float*>(table);
    p.nb = num_buckets;
    p.R = R;
    p.t5 = t5;
    p.dbias = static_cast<float*>(dtable);
  } else if (mode == RELPOS_SHAW) {
    p.aK = static_cast<const __nv_bfloat16*>(table);
    p.aV = static_cast<const __nv_bfloat16*>(table1);
    p.kc = max_distance;
    p.nr = nr;
    float* sh = scratch + n_acc + n_stats;  // every part a multiple of 128 floats
    p.shEnds = sh;
    p.shT = sh + 4 * n_rows;
    p.shU = p.shT + n_rows * nr;
    p.shBP = p.shU + n_rows * nr;
    p.shBdS = p.shBP + n_rows * nr;
    p.shPart = p.shBdS + n_rows * nr;
    p.daK = static_cast<float*>(dtable);
    p.daV = static_cast<float*>(dtable1);
    p.Qp = static_cast<const __nv_bfloat16*>(Q);
    p.dOp = static_cast<const __nv_bfloat16*>(dO);
  } else if (mode == RELPOS_DEBERTA) {
    p.kc = max_distance;
    p.band = reinterpret_cast<const __nv_bfloat16*>(scratch + o_band);
    p.band_pitch = band_pitch;
    p.c2p_const = scratch + o_c2p;
    p.const_pitch = lq_pad;
    p.p2c_ends = scratch + o_ends;
    p.ends_pitch = lk_pad;
    p.dSQ = reinterpret_cast<__nv_bfloat16*>(scratch + o_dsq);
    p.dSK = reinterpret_cast<__nv_bfloat16*>(scratch + o_dsk);
    p.lk_pad = lk_pad;
    p.rowfar = scratch + o_rowfar;
    p.keyfar = scratch + o_keyfar;
    p.dKacc = scratch + o_dk;
    p.rowm1 = scratch + o_m1;
    p.keymk = scratch + o_mk;
    p.shEnds = scratch + o_e4;
    p.Qp = static_cast<const __nv_bfloat16*>(Q);
    p.Kp = static_cast<const __nv_bfloat16*>(K);
    p.Pk = static_cast<const __nv_bfloat16*>(table);
    p.Pq = static_cast<const __nv_bfloat16*>(table1);
    p.dPk = static_cast<float*>(dtable);
    p.dPq = static_cast<float*>(dtable1);
    // the logit scale is 1 / sqrt(3 d)
    p.scale = 1.0f / std::sqrt(static_cast<float>(3 * d));
    p.scale_log2 = p.scale * kLog2e;
    // the gathered dS starts at zero (entries whose key lies outside the
    // keys, or that no visible score reaches, stay so); then the band
    // pre-pass of the forward
    if (cudaMemsetAsync(p.dSQ, 0, BH * lq_pad * k2 * 2, s) != cudaSuccess ||
        cudaMemsetAsync(p.dSK, 0, BH * lk_pad * k2 * 2, s) != cudaSuccess ||
        cudaMemsetAsync(p.rowm1, 0, (r64(BH * lq_pad) + BH * lk_pad) * 4, s) != cudaSuccess)
      return done(RELPOS_ERR_CUDA);
    BandParams bp;
    std::memset(&bp, 0, sizeof(bp));
    bp.BH = static_cast<int>(BH);
    bp.H = H;
    bp.k = max_distance;
    bp.Lq = Lq;
    bp.Lk = Lk;
    bp.q_offset = q_offset;
    bp.scale = p.scale_log2;
    bp.K = static_cast<const __nv_bfloat16*>(K);
    bp.Pq = static_cast<const __nv_bfloat16*>(table1);
    bp.band = reinterpret_cast<__nv_bfloat16*>(scratch + o_band);
    bp.band_pitch = band_pitch;
    bp.c2p_const = scratch + o_c2p;
    bp.const_pitch = lq_pad;
    bp.ends = scratch + o_ends;
    bp.ends_pitch = lk_pad;
    bp.status = status;
    CUtensorMap tpk, tpq;
    if (!make_tmap_table(&tpk, table, H, static_cast<int>(k2)) || !make_tmap_table(&tpq, table1, H, static_cast<int>(k2)))
      return done(RELPOS_ERR_CUDA);
    if (launch_deberta_band(tq, tk, tpk, tpq, bp, s) != cudaSuccess) return done(RELPOS_ERR_CUDA);
  } else {
    p.slopes = static_cast<const float*>(table);
    p.dslopes = static_cast<float*>(dtable);
  }
  p.dQacc = scratch;
  p.lse = scratch + n_acc;  // n_acc is a multiple of 64 floats: 256-byte aligned
  p.Dr = scratch + n_acc + BH * lq_pad;
  p.lq_pad = lq_pad;
  p.dQ = static_cast<__nv_bfloat16*>(dQ);
  p.dK = static_cast<__nv_bfloat16*>(dK);
  p.dV = static_cast<__nv_bfloat16*>(dV);
  p.status = status;
  if (launch_bwd(mode, tq, tk, tv, tdo, tacc, p, s) != cudaSuccess) return done(RELPOS_ERR_CUDA);
  return done(RELPOS_OK);
}

}  // namespace
}  // namespace relpos

extern "C" int relpos_t5_attn_bwd(const void* Q, const void* K, const void* V, const void* dO,
                                  const void* bias, int B, int H, int Lq, int Lk, int d, int num_buckets,
                                  int max_distance, int causal, int q_offset, void* dQ, void* dK, void* dV,
                                  void* dbias, void* stream) {
  return attn_bwd_impl(RELPOS_T5, Q, K, V, dO, bias, nullptr, B, H, Lq, Lk, d, num_buckets, max_distance, causal,
                       q_offset, dQ, dK, dV, dbias, nullptr, stream);
}

extern "C" int relpos_shaw_attn_bwd(const void* Q, const void* K, const void* V, const void* dO,
                                    const void* aK, const void* aV, int B, int H, int Lq, int Lk, int d,
                                    int clip_k, int causal, int q_offset, void* dQ, void* dK, void* dV,
                                    void* daK, void* daV, void* stream) {
  return attn_bwd_impl(RELPOS_SHAW, Q, K, V, dO, aK, aV, B, H, Lq, Lk, d, 0, clip_k, causal, q_offset, dQ, dK,
                       dV, daK, daV, stream);
}

extern "C" int relpos_deberta_attn_bwd(const void* Q, const void* K, const void* V, const void* dO,
                                       const void* Pk, const void* Pq, int B, int H, int Lq, int Lk, int d,
                                       int k, int causal, int q_offset, void* dQ, void* dK, void* dV, void* dPk,
                                       void* dPq, void* stream) {
  return attn_bwd_impl(RELPOS_DEBERTA, Q, K, V, dO, Pk, Pq, B, H, Lq, Lk, d, 0, k, causal, q_offset, dQ, dK, dV,
                       dPk, dPq, stream);
}

extern "C" int relpos_alibi_attn_bwd(const void* Q, const void* K, const void* V, const void* dO,
                                     const void* slopes, int B, int H, int Lq, int Lk, int d, int causal,
                                     int q_offset, void* dQ, void* dK, void* dV, void* dslopes,
                                     void* stream) {
  return attn_bwd_impl(RELPOS_ALIBI, Q, K, V, dO, slopes, nullptr, B, H, Lq, Lk, d, 0, 0, causal, q_offset, dQ,
                       dK, dV, dslopes, nullptr, stream);
}
