// us_internal.h -- host-side declarations shared by the libus translation units.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include "../../include/us.h"

struct UsKParams;

namespace us {

// encoder (us_encode.cu)
size_t encode_pack_smem(int TM, int TK, int elem);
us_status launch_encode(const void* W, int64_t ldw, int M, int K, int TM, int TK, int elem, int order,
                        uint64_t* bitmap, uint32_t* tile_off, void* values, size_t values_cap,
                        uint32_t* counts, unsigned* status, cudaStream_t st);

// generic CUDA-core SpMM (us_spmm.cu); p.split / p.tok_block already chosen
us_status launch_spmm_generic(const UsKParams& p, int elem, cudaStream_t st);
// bytes of partials + counters the generic kernel needs for this launch shape
size_t spmm_generic_ws(int M, int TM, int N, int split, int tok_block);
int spmm_generic_tok_block(int N);

// W4A4 CUDA-core decode kernel for small N (us_w4a4.cu)
bool w4a4_fast_supported(int TM, int TK, int N);
us_status launch_w4a4_fast(const UsKParams& p, cudaStream_t st);
size_t w4a4_fast_ws(int M, int TM, int N, int split);
int w4a4_fast_target_ctas();
int w4a4_fast_tok_block(int N);
int w4a4_fast_max_split();

// W4A4 CUDA-core kernel over a balanced partition of the tile sequence
// (us_w4a4_sk.cu); launch_w4a4_sk takes p.ws = start of the workspace
bool w4a4_sk_supported(int TM, int TK, int M, int K, int N);
size_t w4a4_sk_ws(int M, int K, int N);
int w4a4_sk_variant(int N);   // 0: dp4a consumer, else the mma consumer's 8-token blocks
us_status launch_w4a4_sk(UsKParams p, cudaStream_t st);
// the same kernel on IE-BME 16 x 64 local tiles with areas (us_w4a4_sk_ie.cu);
// p.nTM counts 64-row bands there
bool w4a4_sk_ie_supported(int M, int K, int TM, int TK, int RA, int CA, int N);
size_t w4a4_sk_ie_ws(int M, int K, int N);
us_status launch_w4a4_sk_ie(UsKParams p, cudaStream_t st);

// tensor-core fp16 SpMM for many tokens (us_tc.cu)
bool tc_f16_supported(int TM, int TK, int M, int N);
int tc_tok_block(int N);
int tc_split(int M, int N, int nTK);
int tc_max_split();                  // K slices of one output tile form one cluster
size_t tc_ws(int M, int N, int split);
us_status launch_tc_f16(const UsKParams& p, cudaStream_t st);
// the driver's cuTensorMapEncodeTiled (nullptr if the driver lacks it)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder();

// fp16 SpMM for 1-63 tokens on 64 x 64 row-scan tiles (us_f16_dec.cu)
bool f16_dec_supported(int TM, int TK, int order, int N);
int f16_dec_tok_block(int N);
bool f16_dec_fits(int nTK, int split, int N);
int f16_dec_split(int nTM, int nTK, int N);
us_status launch_f16_dec(const UsKParams& p, cudaStream_t st);


// spMspV (us_spmspv.cu)
us_status launch_spmspv(const UsKParams& p, cudaStream_t st);
us_status launch_encode_ie(const void* W, int64_t ldw, int M, int K, int TM, int TK, int RA, int CA, int elem,
                           const uint8_t* perm, uint64_t* bitmap, uint32_t* tile_off, void* values,
                           size_t values_cap, uint32_t* counts, unsigned* status, cudaStream_t st);
us_status launch_colinfo(const uint64_t* bitmap, int TM, int TK, int64_t nT, uint32_t* colinfo, cudaStream_t st);
us_status launch_spmspv_ci(const UsKParams& p, const uint32_t* colinfo, cudaStream_t st);
size_t spmspv_ws(int M, int TM, int split);
int spmspv_max_split();
// streamed spMspV on 64 x 64 tiles (us_spmspv_stream.cu): its K split, 0 when
// the shape is not supported
int spmspv_stream_split(int TM, int TK, int nTM, int nTK);
us_status launch_spmspv_stream(UsKParams p, cudaStream_t st);

// per-token int4 quantisation of fp16 activations (us_quant.cu)
us_status launch_quantize_x(const uint16_t* X, int N, int K, uint8_t* Xq, uint16_t* s_x, cudaStream_t st);

// device properties of the current device (cached)
int num_sms();

}  // namespace us
