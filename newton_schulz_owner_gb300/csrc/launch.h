// Host-side launchers shared between the C-ABI layer and the kernel files.
#pragma once
#include <cstddef>
#include <cuda_runtime.h>

#include "tables.h"

namespace dm {

// Every successful kernel launch of the library is counted per host thread
// (read through dmuon_launch_count).
void note_launch(int kernels = 1);
inline cudaError_t counted(cudaError_t e) {
  if (e == cudaSuccess) note_launch();
  return e;
}

// ns_gemm.cu
size_t ns_gemm_smem_bytes();
// Once per device: opt into large shared memory and find how many CTA pairs
// (clusters of two) can be resident at once.
cudaError_t ns_gemm_prepare(int num_sms, int* max_clusters);
cudaError_t launch_ns_gemm(const GemmArgs& g, int kind, int max_clusters, cudaStream_t s);
// Product-launch tracing: while active, every product launch on `device` that
// still fits writes one TraceRec per CTA into `buf` (room for `records`).
void trace_begin(void* buf, size_t records, int device);
long long trace_end();  // stops tracing; returns the records handed out
// Per-matrix diagonal shift b*s + c*s^2 with s = trace(A)/m, A = slot `slot`.
cudaError_t launch_diag_shift(const Bucket* buckets, int n_buckets, int first_internal,
                              int n_mats, int slot, float b, float c, float* shift,
                              cudaStream_t s);

// elementwise.cu
// Copy `bytes` (multiple of 16) from host memory into device memory through
// kernel parameters (stream-ordered, no host staging, no allocation).
cudaError_t launch_upload(void* dst, const void* src, size_t bytes, cudaStream_t s);
// A contiguous range of the per-matrix table: ew[0, n) are entries first ..
// first + n - 1 (device pointer to entry `first`); the kernel works on the
// elementwise chunks [chunk_base, chunk_base + chunks) of those matrices.
struct EwRange {
  const EwMat* ew;
  int n, first;
  long long chunk_base, chunks;
};
cudaError_t launch_momentum_pack(const EwRange& r, bool grad_bf16, float beta,
                                 __nv_bfloat16* packed, float* partials, cudaStream_t s);
cudaError_t launch_norm_partials(const EwRange& r, const __nv_bfloat16* packed, float* partials,
                                 cudaStream_t s);
cudaError_t launch_norm_finalize(const EwRange& r, const float* partials, float eps,
                                 float* inv_norm, cudaStream_t s);
cudaError_t launch_relayout(const EwRange& r, const __nv_bfloat16* packed, const float* inv_norm,
                            cudaStream_t s);
cudaError_t launch_scale_inplace(const EwRange& r, __nv_bfloat16* packed, const float* inv_norm,
                                 cudaStream_t s);
cudaError_t launch_update(const EwRange& r, bool weight_bf16, float lr,
                          const __nv_bfloat16* packed, cudaStream_t s);
cudaError_t launch_wait_timeout(int* err, long long budget_cycles, cudaStream_t s);
cudaError_t launch_adamw(const AdamTensor* ts, int n, long long total_chunks, bool p_bf16,
                         bool g_bf16, const AdamScalars& k, cudaStream_t s);

}  // namespace dm
