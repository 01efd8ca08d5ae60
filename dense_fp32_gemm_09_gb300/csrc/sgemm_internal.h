// Host-side declarations shared by the dispatcher and the kernel translation
// units; the types the kernels themselves see are in sgemm_args.h.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/sgemm.h"
#include "sgemm_args.h"

namespace sgemm {

// Device status word (sgemm_status.cu): address on the current device, and a
// synchronous read-and-clear of its value.
int* status_word_ptr();
int read_and_clear_status(int* value);
int run_wait_selftest(int limit_ms);

// Sums the partial tiles of a stream-K launch into C (sgemm_reduce.cu).  Launch
// it on the same stream right after the main kernel when a.sk_tiles > 0.
cudaError_t launch_sk_reduce(const GemmArgs& a, int bm, int bn, int sms, cudaStream_t stream);
int reduce_chunks(int bm, int bn, int sk_tiles, int sms);

// Sets the text sgemm_last_error() returns on this thread: a plain message, or
// "<what>: <CUDA error name> (<description>)".
void set_last_error_message(const char* msg);
void set_cuda_error(const char* what, cudaError_t e);

// SGEMM_ERR_UNSUPPORTED (with a message) when M, N or K is above 2^30, else SGEMM_OK.
int check_sizes(int M, int N, int K);

// Argument checks of the public entry points (sizes, leading dimensions of the
// stored operands, null pointers, C overlapping A or B); op = 1 means the operand
// is stored transposed.  SGEMM_OK, SGEMM_ERR_INVALID_ARG with a message, or
// SGEMM_ERR_UNSUPPORTED for a dimension above 2^30.
int check_operands(int transa, int transb, int M, int N, int K, const float* A, int lda,
                   const float* B, int ldb, const float* C, int ldc);

// Destroys the host-buffer entry point's streams and events (sgemm_shutdown).
void shutdown_host_pipes();

// Forgets which devices had the 3xTF32 kernels' shared-memory limit raised
// (sgemm_shutdown): the next launch on each device sets it again.
void forget_tf32x3_attributes();

// Drops the cached device addresses of sgemm_run_noalloc's static scratch
// (sgemm_shutdown); the next call looks them up again.
void forget_noalloc_scratch();

// 3xTF32 tensor-core path (sgemm_tf32x3.cu).
size_t tf32x3_workspace_bytes(int M, int N, int K);
// write_ahi = false leaves the Ahi region unwritten: the multiply then takes hi
// from A itself (a_hi = A, lda_hi = lda; A 16-byte aligned with lda % 4 == 0).
int tf32x3_prepare(int M, int N, int K, const float* A, long long lda, const float* B,
                   long long ldb, void* ws, size_t ws_bytes, int sms, cudaStream_t stream,
                   bool write_ahi = true);
int tf32x3_multiply(int M, int N, int K, float alpha, float beta, float* C, long long ldc,
                    int c_vec, void* ws, size_t ws_bytes, int sms, cudaStream_t stream,
                    int* launches, const float* a_hi = nullptr, long long lda_hi = 0);
int tf32x3_tile_width(int M, int N, int K, int sms);
int tf32x3_query(int M, int N, int K, int sms, sgemm_config* out);


}  // namespace sgemm
