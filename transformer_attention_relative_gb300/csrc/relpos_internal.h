// relpos_internal.h -- launchers shared between the library's translation units.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <cstddef>
#include <cstdint>

#include "relpos_common.cuh"

namespace relpos {

uint32_t fwd_smem_bytes(int mode, const FwdParams& p);
uint32_t fwd_max_smem_bytes();
int fwd_num_items(const FwdParams& p);
// How many trailing pair items (of npair_items, with BH items per pair row)
// to run as two split items each on a grid of num_sms persistent CTAs.
int fwd_split_items(int npair_items, int BH, int Lq, int causal, int num_sms);
// tmS: Transformer-XL's key sinusoid table (unused by the other modes)
cudaError_t launch_fwd(int mode, bool out_f32, const CUtensorMap& tmQ, const CUtensorMap& tmK,
                       const CUtensorMap& tmV, const CUtensorMap& tmS, const FwdParams& p, int num_sms,
                       cudaStream_t stream);

// T5 bucket thresholds for offsets up to nmax (see api.cu) and the shared
// relative-parameter checks; both return RELPOS_* codes.
int t5_setup(int num_buckets, int max_distance, int causal, long long nmax, T5Index* ix, int* R);
int check_rel_params(int mode, int num_buckets, int rel_param, int causal);

cudaError_t launch_deberta_band(const CUtensorMap& tmQ, const CUtensorMap& tmK, const CUtensorMap& tmPk,
                                const CUtensorMap& tmPq, const BandParams& bp, cudaStream_t stream);

cudaError_t launch_txl_prep(const TxlParams& p, cudaStream_t stream);
// T5 forward over keys at explicit positions through the fused kernel (any
// number of query rows; the C ABI's positions entry point takes it beyond the
// decode kernel's rows)
int attn_fwd_t5_positions(const void* Q, const void* K, const void* V, const void* bias, const int* key_pos,
                          int B, int H, int Lq, int Lk, int num_buckets, int max_distance, int causal,
                          int q_offset, void* out, void* stream);

int decode_chunk_keys();
cudaError_t launch_decode(const DecodeParams& p, cudaStream_t stream);
// Floats of per-chunk partials (64 output values, max, sum) the split-key
// decode needs for `rows` query rows over Lk keys.
size_t decode_partial_floats(size_t rows, int Lk);
// The decode kernels' parameter block; `part` holds decode_partial_floats()
// floats, key_pos is null for keys at positions 0 .. Lk - 1.
DecodeParams make_decode_params(const void* Q, const void* K, const void* V, const void* bias,
                                const int* key_pos, int B, int H, int Lq, int Lk, int causal,
                                int q_offset, float scale_log2, const T5Index& t5, int R,
                                float* part, void* out, bool out_f32);

// true when p is 16-byte aligned (the kernels' vector loads and stores)
bool aligned16(const void* p);

}  // namespace relpos
