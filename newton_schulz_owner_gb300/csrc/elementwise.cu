// Memory-bound kernels of the owner-side Muon step.
//
//   momentum_pack   M <- beta*M + (1-beta)*G;  U = (1-beta)*G + beta*M;
//                   packed <- bf16(U); per-chunk fp32 partial sums of U^2
//   norm_partials   the same partial sums from bf16 values already packed
//   norm_finalize   inv_i = 1 / (sqrt(sum of matrix i's partials) + eps), fp64
//   relayout        X0 = U * inv into the working layout (the parameter's own
//                   orientation, rows padded to the slot pitch): a chunked copy
//   scale_inplace   packed <- bf16(U * inv)  (ns_steps = 0)
//   update          W <- W - lr * sqrt(max(1, rows/cols)) * O
// Every kernel reads and writes 16-byte vectors where the pointers allow and
// reduces in a fixed order, so results are bit-reproducible.
#include "dmuon.h"
#include "launch.h"
#include "ptx.cuh"
#include "tables.h"

#include <cuda_bf16.h>

namespace dm {
namespace {

constexpr int kVec = 8;                                   // elements per thread step
constexpr int kIters = kChunk / (kVec * kEwThreads);      // 4
static_assert(kChunk == kVec * kEwThreads * kIters, "chunk shape");

// Largest i with ew[i].chunk_begin <= chunk (ew sorted by chunk_begin).
DM_DEV int find_mat(const EwMat* ew, int n, long long chunk) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (ew[mid].chunk_begin <= chunk) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

DM_DEV void bf16x8_to_f32(uint4 u, float (&f)[8]) {
  const uint32_t w[4] = {u.x, u.y, u.z, u.w};
#pragma unroll
  for (int k = 0; k < 4; ++k) {
    const float2 t = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[k]));
    f[2 * k] = t.x;
    f[2 * k + 1] = t.y;
  }
}

DM_DEV uint32_t f32x2_to_bf16x2(float a, float b) {
  __nv_bfloat162 t = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&t);
}

DM_DEV uint4 f32x8_to_bf16x8(const float (&f)[8]) {
  uint4 u;
  u.x = f32x2_to_bf16x2(f[0], f[1]);
  u.y = f32x2_to_bf16x2(f[2], f[3]);
  u.z = f32x2_to_bf16x2(f[4], f[5]);
  u.w = f32x2_to_bf16x2(f[6], f[7]);
  return u;
}

// Fixed-order block sum (warp xor-tree, then warp totals in warp order).
DM_DEV float block_sum(float v) {
  __shared__ float warp_tot[kEwThreads / 32];
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) warp_tot[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
  if (threadIdx.x == 0)
    for (int w = 0; w < kEwThreads / 32; ++w) s += warp_tot[w];
  return s;  // valid in thread 0
}

// Every chunked kernel below works on the sub-range ew[0, n) of the per-matrix
// table; `base` is the global index of its first chunk.
template <bool G_BF16>
__global__ void __launch_bounds__(kEwThreads) momentum_pack_kernel(const EwMat* __restrict__ ew,
                                                                   int n, long long base,
                                                                   float beta,
                                                                   __nv_bfloat16* packed,
                                                                   float* partials) {
  const long long chunk = base + blockIdx.x;
  const EwMat& E = ew[find_mat(ew, n, chunk)];
  const long long start = (chunk - E.chunk_begin) * kChunk;
  const long long end = min(E.numel, start + kChunk);
  const float omb = 1.f - beta;
  const bool vec = (E.flags & kFlagVecGM) != 0;
  __nv_bfloat16* P = packed + E.packed_off;
  float* Mo = E.mom;
  float ss = 0.f;
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const long long e = start + (long long)(it * kEwThreads + threadIdx.x) * kVec;
    if (e >= end) break;
    float g[kVec], m[kVec], u[kVec];
    const bool full = vec && e + kVec <= end;
    if (full) {
      if (G_BF16) {
        bf16x8_to_f32(*reinterpret_cast<const uint4*>(
                          reinterpret_cast<const __nv_bfloat16*>(E.g) + e), g);
      } else {
        const float4* gp = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(E.g) + e);
        const float4 a = gp[0], b = gp[1];
        g[0] = a.x; g[1] = a.y; g[2] = a.z; g[3] = a.w;
        g[4] = b.x; g[5] = b.y; g[6] = b.z; g[7] = b.w;
      }
      const float4* mp = reinterpret_cast<const float4*>(Mo + e);
      const float4 a = mp[0], b = mp[1];
      m[0] = a.x; m[1] = a.y; m[2] = a.z; m[3] = a.w;
      m[4] = b.x; m[5] = b.y; m[6] = b.z; m[7] = b.w;
    } else {
#pragma unroll
      for (int k = 0; k < kVec; ++k) {
        const bool in = e + k < end;
        g[k] = !in ? 0.f
                   : (G_BF16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(E.g)[e + k])
                             : reinterpret_cast<const float*>(E.g)[e + k]);
        m[k] = in ? Mo[e + k] : 0.f;
      }
    }
#pragma unroll
    for (int k = 0; k < kVec; ++k) {
      const float gg = omb * g[k];
      m[k] = fmaf(beta, m[k], gg);
      u[k] = fmaf(beta, m[k], gg);
    }
    if (full) {
      float4* mp = reinterpret_cast<float4*>(Mo + e);
      mp[0] = make_float4(m[0], m[1], m[2], m[3]);
      mp[1] = make_float4(m[4], m[5], m[6], m[7]);
#pragma unroll
      for (int k = 0; k < kVec; ++k) ss = fmaf(u[k], u[k], ss);
      *reinterpret_cast<uint4*>(P + e) = f32x8_to_bf16x8(u);
    } else {
#pragma unroll
      for (int k = 0; k < kVec; ++k) {
        if (e + k < end) {
          Mo[e + k] = m[k];
          P[e + k] = __float2bfloat16_rn(u[k]);
          ss = fmaf(u[k], u[k], ss);
        }
      }
    }
  }
  const float tot = block_sum(ss);
  if (threadIdx.x == 0) partials[E.partial_begin + (chunk - E.chunk_begin)] = tot;
}

__global__ void __launch_bounds__(kEwThreads) norm_partials_kernel(const EwMat* __restrict__ ew,
                                                                   int n, long long base,
                                                                   const __nv_bfloat16* packed,
                                                                   float* partials) {
  const long long chunk = base + blockIdx.x;
  const EwMat& E = ew[find_mat(ew, n, chunk)];
  const long long start = (chunk - E.chunk_begin) * kChunk;
  const long long end = min(E.numel, start + kChunk);
  const __nv_bfloat16* P = packed + E.packed_off;
  float ss = 0.f;
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const long long e = start + (long long)(it * kEwThreads + threadIdx.x) * kVec;
    if (e >= end) break;
    if (e + kVec <= end) {
      float u[kVec];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(P + e), u);
#pragma unroll
      for (int k = 0; k < kVec; ++k) ss = fmaf(u[k], u[k], ss);
    } else {
      for (int k = 0; k < kVec; ++k)
        if (e + k < end) {
          const float u = __bfloat162float(P[e + k]);
          ss = fmaf(u, u, ss);
        }
    }
  }
  const float tot = block_sum(ss);
  if (threadIdx.x == 0) partials[E.partial_begin + (chunk - E.chunk_begin)] = tot;
}

__global__ void __launch_bounds__(kEwThreads) norm_finalize_kernel(const EwMat* __restrict__ ew,
                                                                   const float* partials,
                                                                   float eps, float* inv_norm) {
  __shared__ double red[kEwThreads];
  const EwMat& E = ew[blockIdx.x];
  double s = 0.0;
  for (int c = threadIdx.x; c < E.n_chunks; c += kEwThreads)
    s += (double)partials[E.partial_begin + c];
  red[threadIdx.x] = s;
  __syncthreads();
  for (int w = kEwThreads / 2; w > 0; w >>= 1) {
    if (threadIdx.x < w) red[threadIdx.x] += red[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) inv_norm[blockIdx.x] = (float)(1.0 / (sqrt(red[0]) + (double)eps));
}

// X0 = U * inv into the working layout: the parameter's own orientation with
// rows padded to the slot pitch.  One block per chunk of the packed matrix, read
// in its row-major order like every other chunked kernel; where cols % 8 == 0
// each thread moves 16-byte vectors, none of which crosses a row, to
// row * pitch + col.
__global__ void __launch_bounds__(kEwThreads) relayout_kernel(const EwMat* __restrict__ ew, int n,
                                                              long long base,
                                                              const __nv_bfloat16* packed,
                                                              const float* inv_norm) {
  const long long chunk = base + blockIdx.x;
  const int i = find_mat(ew, n, chunk);
  const EwMat& E = ew[i];
  const long long start = (chunk - E.chunk_begin) * kChunk;
  const long long end = min(E.numel, start + kChunk);
  const float inv = inv_norm[i];
  const __nv_bfloat16* P = packed + E.packed_off;
  __nv_bfloat16* X = E.x0;
  const long long cols = E.cols, pitch = E.pitch_x;
  if (E.flags & kFlagRowsAligned) {
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
      const long long e = start + (long long)(it * kEwThreads + threadIdx.x) * kVec;
      if (e >= end) break;
      const long long r = e / cols, c = e - r * cols;
      float f[kVec];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(P + e), f);
#pragma unroll
      for (int k = 0; k < kVec; ++k) f[k] *= inv;
      *reinterpret_cast<uint4*>(X + r * pitch + c) = f32x8_to_bf16x8(f);
    }
  } else {
#pragma unroll
    for (int it = 0; it < kIters; ++it) {
      const long long e0 = start + (long long)(it * kEwThreads + threadIdx.x) * kVec;
      if (e0 >= end) break;
      for (int k = 0; k < kVec && e0 + k < end; ++k) {
        const long long e = e0 + k, r = e / cols, c = e - r * cols;
        X[r * pitch + c] = __float2bfloat16_rn(__bfloat162float(P[e]) * inv);
      }
    }
  }
}

__global__ void __launch_bounds__(kEwThreads) scale_inplace_kernel(const EwMat* __restrict__ ew,
                                                                   int n, long long base,
                                                                   __nv_bfloat16* packed,
                                                                   const float* inv_norm) {
  const long long chunk = base + blockIdx.x;
  const int i = find_mat(ew, n, chunk);
  const EwMat& E = ew[i];
  const long long start = (chunk - E.chunk_begin) * kChunk;
  const long long end = min(E.numel, start + kChunk);
  const float inv = inv_norm[i];
  __nv_bfloat16* P = packed + E.packed_off;
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const long long e = start + (long long)(it * kEwThreads + threadIdx.x) * kVec;
    if (e >= end) break;
    if (e + kVec <= end) {
      float u[kVec];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(P + e), u);
#pragma unroll
      for (int k = 0; k < kVec; ++k) u[k] *= inv;
      *reinterpret_cast<uint4*>(P + e) = f32x8_to_bf16x8(u);
    } else {
      for (int k = 0; k < kVec; ++k)
        if (e + k < end) P[e + k] = __float2bfloat16_rn(__bfloat162float(P[e + k]) * inv);
    }
  }
}

template <bool W_BF16>
__global__ void __launch_bounds__(kEwThreads) update_kernel(const EwMat* __restrict__ ew, int n,
                                                            long long base, float lr,
                                                            const __nv_bfloat16* packed) {
  const long long chunk = base + blockIdx.x;
  const EwMat& E = ew[find_mat(ew, n, chunk)];
  const long long start = (chunk - E.chunk_begin) * kChunk;
  const long long end = min(E.numel, start + kChunk);
  const float coef = -(lr * E.upd_scale);
  const bool vec = (E.flags & kFlagVecW) != 0;
  const __nv_bfloat16* P = packed + E.packed_off;
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const long long e = start + (long long)(it * kEwThreads + threadIdx.x) * kVec;
    if (e >= end) break;
    if (vec && e + kVec <= end) {
      float o[kVec], w[kVec];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(P + e), o);
      if (W_BF16) {
        uint4* wp = reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(E.w) + e);
        bf16x8_to_f32(*wp, w);
#pragma unroll
        for (int k = 0; k < kVec; ++k) w[k] = fmaf(coef, o[k], w[k]);
        *wp = f32x8_to_bf16x8(w);
      } else {
        float4* wp = reinterpret_cast<float4*>(reinterpret_cast<float*>(E.w) + e);
        const float4 a = wp[0], b = wp[1];
        wp[0] = make_float4(fmaf(coef, o[0], a.x), fmaf(coef, o[1], a.y), fmaf(coef, o[2], a.z),
                            fmaf(coef, o[3], a.w));
        wp[1] = make_float4(fmaf(coef, o[4], b.x), fmaf(coef, o[5], b.y), fmaf(coef, o[6], b.z),
                            fmaf(coef, o[7], b.w));
      }
    } else {
      for (int k = 0; k < kVec; ++k) {
        if (e + k >= end) break;
        const float o = __bfloat162float(P[e + k]);
        if (W_BF16) {
          __nv_bfloat16* wp = reinterpret_cast<__nv_bfloat16*>(E.w) + e + k;
          *wp = __float2bfloat16_rn(fmaf(coef, o, __bfloat162float(*wp)));
        } else {
          float* wp = reinterpret_cast<float*>(E.w) + e + k;
          *wp = fmaf(coef, o, *wp);
        }
      }
    }
  }
}

DM_DEV int find_adam(const AdamTensor* t, int n, long long chunk) {
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (t[mid].chunk_begin <= chunk) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

template <bool BF16>
DM_DEV void load8(const void* base, long long e, float (&f)[8]) {
  if (BF16) {
    bf16x8_to_f32(*reinterpret_cast<const uint4*>(reinterpret_cast<const __nv_bfloat16*>(base) + e),
                  f);
  } else {
    const float4* q = reinterpret_cast<const float4*>(reinterpret_cast<const float*>(base) + e);
    const float4 a = q[0], b = q[1];
    f[0] = a.x; f[1] = a.y; f[2] = a.z; f[3] = a.w;
    f[4] = b.x; f[5] = b.y; f[6] = b.z; f[7] = b.w;
  }
}

template <bool BF16>
DM_DEV float load1(const void* base, long long e) {
  return BF16 ? __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(base)[e])
              : reinterpret_cast<const float*>(base)[e];
}

DM_DEV void store8f(float* base, long long e, const float (&f)[8]) {
  float4* q = reinterpret_cast<float4*>(base + e);
  q[0] = make_float4(f[0], f[1], f[2], f[3]);
  q[1] = make_float4(f[4], f[5], f[6], f[7]);
}

// AdamW with decoupled weight decay, fp32 arithmetic:
//   p <- p * decay;  m <- b1 m + (1-b1) g;  v <- b2 v + (1-b2) g^2;
//   p <- p - step_size * m / (sqrt(v) * inv_bc2_sqrt + eps)
// At most 64 registers where that needs no spills (bf16 parameter or
// gradient), so that four blocks fit on an SM: with seven streams per element
// the kernel needs many loads in flight to cover DRAM latency.
template <bool P_BF16, bool G_BF16>
__global__ void __launch_bounds__(kEwThreads, (P_BF16 || G_BF16) ? 4 : 3)
    adamw_kernel(const AdamTensor* __restrict__ ts, int n, AdamScalars ks) {
  const long long chunk = blockIdx.x;
  const AdamTensor T = ts[find_adam(ts, n, chunk)];
  const long long start = (chunk - T.chunk_begin) * kChunk;
  const long long end = min(T.numel, start + kChunk);
  const float b1 = ks.b1, b2 = ks.b2, omb1 = ks.omb1, omb2 = ks.omb2;
  const float decay = ks.decay, step_size = ks.step_size, inv_bc2_sqrt = ks.inv_bc2_sqrt;
  const float eps = ks.eps;
#pragma unroll
  for (int it = 0; it < kIters; ++it) {
    const long long e = start + (long long)(it * kEwThreads + threadIdx.x) * kVec;
    if (e >= end) break;
    if (T.vec && e + kVec <= end) {
      float p[kVec], g[kVec], m[kVec], v[kVec];
      load8<P_BF16>(T.p, e, p);
      load8<G_BF16>(T.g, e, g);
      load8<false>(T.m, e, m);
      load8<false>(T.v, e, v);
#pragma unroll
      for (int k = 0; k < kVec; ++k) {
        m[k] = fmaf(b1, m[k], omb1 * g[k]);
        v[k] = fmaf(b2, v[k], omb2 * g[k] * g[k]);
        const float denom = fmaf(sqrtf(v[k]), inv_bc2_sqrt, eps);
        p[k] = fmaf(-step_size, m[k] / denom, p[k] * decay);
      }
      store8f(T.m, e, m);
      store8f(T.v, e, v);
      if (P_BF16)
        *reinterpret_cast<uint4*>(reinterpret_cast<__nv_bfloat16*>(T.p) + e) = f32x8_to_bf16x8(p);
      else
        store8f(reinterpret_cast<float*>(T.p), e, p);
    } else {
      for (int k = 0; k < kVec && e + k < end; ++k) {
        const long long i = e + k;
        const float g = load1<G_BF16>(T.g, i);
        const float m = fmaf(b1, T.m[i], omb1 * g);
        const float v = fmaf(b2, T.v[i], omb2 * g * g);
        const float denom = fmaf(sqrtf(v), inv_bc2_sqrt, eps);
        const float p = fmaf(-step_size, m / denom, load1<P_BF16>(T.p, i) * decay);
        T.m[i] = m;
        T.v[i] = v;
        if (P_BF16) reinterpret_cast<__nv_bfloat16*>(T.p)[i] = __float2bfloat16_rn(p);
        else reinterpret_cast<float*>(T.p)[i] = p;
      }
    }
  }
}

// Kernel-parameter payload for table uploads (kernel parameters may hold up to
// 32764 bytes).
constexpr int kUploadBytes = 30720;
struct UploadArgs {
  uint4* dst;
  int n16;
  int pad_;
  uint4 data[kUploadBytes / 16];
};

__global__ void upload_kernel(const __grid_constant__ UploadArgs a) {
  for (int k = threadIdx.x; k < a.n16; k += blockDim.x) a.dst[k] = a.data[k];
  // the uploaded tables include TMA tensor maps
  tensormap_release();
}

__global__ void wait_timeout_kernel(int* err, long long budget_cycles) {
  __shared__ uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_barrier_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    // nobody arrives on `bar`: the bounded wait must give up
    if (!mbar_wait(&bar, 0, nullptr, budget_cycles)) atomicCAS(err, 0, int(DMUON_ERR_TIMEOUT));
  }
}

inline unsigned grid_of(long long blocks) { return static_cast<unsigned>(blocks); }

}  // namespace

cudaError_t launch_upload(void* dst, const void* src, size_t bytes, cudaStream_t s) {
  const unsigned char* p = static_cast<const unsigned char*>(src);
  unsigned char* d = static_cast<unsigned char*>(dst);
  UploadArgs a;
  for (size_t off = 0; off < bytes; off += kUploadBytes) {
    const size_t nb = (bytes - off) < size_t(kUploadBytes) ? (bytes - off) : size_t(kUploadBytes);
    a.dst = reinterpret_cast<uint4*>(d + off);
    a.n16 = int(nb / 16);
    a.pad_ = 0;
    memcpy(a.data, p + off, nb);
    upload_kernel<<<1, 256, 0, s>>>(a);
    const cudaError_t e = counted(cudaGetLastError());
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

cudaError_t launch_momentum_pack(const EwRange& r, bool grad_bf16, float beta,
                                 __nv_bfloat16* packed, float* partials, cudaStream_t s) {
  if (r.chunks <= 0) return cudaSuccess;
  if (grad_bf16)
    momentum_pack_kernel<true><<<grid_of(r.chunks), kEwThreads, 0, s>>>(r.ew, r.n, r.chunk_base,
                                                                        beta, packed, partials);
  else
    momentum_pack_kernel<false><<<grid_of(r.chunks), kEwThreads, 0, s>>>(r.ew, r.n, r.chunk_base,
                                                                         beta, packed, partials);
  return counted(cudaGetLastError());
}

cudaError_t launch_norm_partials(const EwRange& r, const __nv_bfloat16* packed, float* partials,
                                 cudaStream_t s) {
  if (r.chunks <= 0) return cudaSuccess;
  norm_partials_kernel<<<grid_of(r.chunks), kEwThreads, 0, s>>>(r.ew, r.n, r.chunk_base, packed,
                                                                partials);
  return counted(cudaGetLastError());
}

cudaError_t launch_norm_finalize(const EwRange& r, const float* partials, float eps,
                                 float* inv_norm, cudaStream_t s) {
  if (r.n <= 0) return cudaSuccess;
  norm_finalize_kernel<<<r.n, kEwThreads, 0, s>>>(r.ew, partials, eps, inv_norm + r.first);
  return counted(cudaGetLastError());
}

cudaError_t launch_relayout(const EwRange& r, const __nv_bfloat16* packed, const float* inv_norm,
                            cudaStream_t s) {
  if (r.chunks <= 0) return cudaSuccess;
  relayout_kernel<<<grid_of(r.chunks), kEwThreads, 0, s>>>(r.ew, r.n, r.chunk_base, packed,
                                                           inv_norm + r.first);
  return counted(cudaGetLastError());
}

cudaError_t launch_scale_inplace(const EwRange& r, __nv_bfloat16* packed, const float* inv_norm,
                                 cudaStream_t s) {
  if (r.chunks <= 0) return cudaSuccess;
  scale_inplace_kernel<<<grid_of(r.chunks), kEwThreads, 0, s>>>(r.ew, r.n, r.chunk_base, packed,
                                                                inv_norm + r.first);
  return counted(cudaGetLastError());
}

cudaError_t launch_update(const EwRange& r, bool weight_bf16, float lr,
                          const __nv_bfloat16* packed, cudaStream_t s) {
  if (r.chunks <= 0) return cudaSuccess;
  if (weight_bf16)
    update_kernel<true><<<grid_of(r.chunks), kEwThreads, 0, s>>>(r.ew, r.n, r.chunk_base, lr,
                                                                 packed);
  else
    update_kernel<false><<<grid_of(r.chunks), kEwThreads, 0, s>>>(r.ew, r.n, r.chunk_base, lr,
                                                                  packed);
  return counted(cudaGetLastError());
}

cudaError_t launch_adamw(const AdamTensor* ts, int n, long long total_chunks, bool p_bf16,
                         bool g_bf16, const AdamScalars& k, cudaStream_t s) {
  if (total_chunks <= 0) return cudaSuccess;
  const unsigned grid = grid_of(total_chunks);
  if (p_bf16 && g_bf16)
    adamw_kernel<true, true><<<grid, kEwThreads, 0, s>>>(ts, n, k);
  else if (p_bf16)
    adamw_kernel<true, false><<<grid, kEwThreads, 0, s>>>(ts, n, k);
  else if (g_bf16)
    adamw_kernel<false, true><<<grid, kEwThreads, 0, s>>>(ts, n, k);
  else
    adamw_kernel<false, false><<<grid, kEwThreads, 0, s>>>(ts, n, k);
  return counted(cudaGetLastError());
}

cudaError_t launch_wait_timeout(int* err, long long budget_cycles, cudaStream_t s) {
  wait_timeout_kernel<<<1, 32, 0, s>>>(err, budget_cycles);
  return counted(cudaGetLastError());
}

}  // namespace dm
