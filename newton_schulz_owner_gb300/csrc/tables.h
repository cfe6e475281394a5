// Device-side tables that the host planner writes into the caller's
// workspace and the kernels read.  Plain-old-data only.
#pragma once
#include <cstdint>
#include <cuda_bf16.h>

namespace dm {

// Elementwise kernels (momentum + pack, norm partials, relayout, update) walk
// each matrix in chunks of kChunk elements of its row-major order; one block
// per chunk.
constexpr int kChunk = 8192;
constexpr int kEwThreads = 256;

// Per-bucket buffers.  Slots 0-1 hold m x n working matrices X, slots 2-7 hold
// m x m matrices (A, B for standard Newton-Schulz; A, P, Q, T for Gram).
constexpr int kSlots = 8;
enum Slot : int { SX0 = 0, SX1 = 1, SM0 = 2, SM1 = 3, SM2 = 4, SM3 = 5, SM4 = 6, SM5 = 7 };
__host__ __device__ constexpr bool slot_is_x(int s) { return s < 2; }
// Two TMA tensor maps per slot: the operand map (64 x 64 boxes, 128-byte
// swizzle) at `slot`, and the epilogue map (32 x 32 boxes, 64-byte swizzle)
// at `kSlots + slot`.
constexpr int kMapsPerBucket = 2 * kSlots;

// EwMat::flags
constexpr int kFlagVecGM = 1;      // grad, momentum 16-byte aligned
constexpr int kFlagVecW = 2;       // weight 16-byte aligned
constexpr int kFlagRowsAligned = 4;  // cols % 8 == 0: packed rows 16-byte aligned

// One entry per caller matrix, in the caller's order.
struct EwMat {
  const void* g;           // gradient (bf16 or fp32)
  float* mom;              // momentum (fp32)
  void* w;                 // weight (bf16 or fp32)
  __nv_bfloat16* x0;       // working-layout destination (bucket slot 0)
  long long packed_off;    // element offset of the packed segment
  long long numel;         // rows * cols
  long long chunk_begin;   // first elementwise chunk
  long long partial_begin; // first norm partial sum: caller order, so that the
                           // partials' layout does not depend on the variant
                           // (a pack and a later Newton-Schulz call may plan
                           // their buckets differently)
  int rows, cols;
  int n_chunks;
  int pitch_x;             // row pitch of the working layout (elements); the layout
                           // keeps the parameter's orientation (Y = X^T when rows > cols)
  int flags;
  float upd_scale;         // sqrt(max(1, rows / cols))
  int active;              // 0 for empty matrices (rows or cols == 0)
};

// Matrices with the same working shape (m, n) and orientation form a bucket;
// each bucket's buffers hold `count` matrices back to back at a fixed stride,
// so one 3-D tensor map per buffer covers the whole bucket.  The m x n slots
// keep the parameter's orientation: X (m x n) for a wide or square parameter,
// Y = X^T (n x m) for a tall one (`tall`).
struct Bucket {
  int m, n, count, first;        // first: internal index of the bucket's first matrix
  int pitch_x, pitch_m;          // row pitch (elements) of X slots / m x m slots
  long long stride_x, stride_m;  // elements between consecutive matrices
  __nv_bfloat16* slot[kSlots];   // base of each slot (null if unused)
  int tmap;                      // index of the bucket's first tensor map (kMapsPerBucket maps)
  int sym_off, sym_count;        // upper-triangle tile list of an m x m product
  int full_ti, full_tj;          // tile grid of an m x n product
  int sym_begin;                 // first tile of this bucket in a symmetric launch
  int full_begin;                // first tile of this bucket in a full launch
  int tall;                      // rows > cols: X slots hold Y = X^T (n rows x m columns)
};

// One tensor of an AdamW group (any shape, contiguous), walked in chunks.
struct AdamTensor {
  void* p;                 // parameter (bf16 or fp32)
  const void* g;           // gradient (bf16 or fp32)
  float* m;                // first moment
  float* v;                // second moment
  long long numel;
  long long chunk_begin;
  int vec;                 // all four pointers 16-byte aligned
  int pad_;
};

// Per-step AdamW scalars, formed in double on the host and rounded once.
struct AdamScalars {
  float b1, b2, omb1, omb2;      // beta1, beta2, 1 - beta1, 1 - beta2
  float step_size;               // lr / (1 - beta1^t)
  float inv_bc2_sqrt;            // 1 / sqrt(1 - beta2^t)
  float eps;
  float decay;                   // 1 - lr * weight_decay
};

// Internal (bucket-major) order -> caller matrix.
struct InternalMat {
  long long packed_off;
  int caller;
  int pad_;
};

// Kinds of product launch; one launch covers buckets of one orientation, so
// the operand layouts and the instruction descriptor are compile-time.
//   kSymK     symmetric L R^T, both operands K-major (wide/square X X^T, m x m products)
//   kSymMN    symmetric Y^T Y of tall buckets, both operands MN-major
//   kFullWide X' = alpha X + gamma L X  (L m x m K-major, X MN-major)
//   kFullTall Y' = alpha Y + gamma Y L  (Y K-major, L symmetric, K-major)
enum ProductKind : int { kSymK = 0, kSymMN = 1, kFullWide = 2, kFullTall = 3 };

// Tile shape of the Newton-Schulz products: a CTA pair computes a 256 x 256
// tile; each CTA holds 128 of its rows (and loads half of its columns'
// operand); one pipeline stage carries kBK = 128 of the reduction dimension.
constexpr int kTileM = 256, kTileN = 256, kCtaM = 128, kBK = 128;

// One record per CTA of a traced product launch (see dmuon_trace_begin):
// %globaltimer nanoseconds at kernel entry, at the leader's first MMA issue,
// after the leader's last MMA completed, and at exit (MMA stamps are 0 in the
// second CTA of a pair and in a CTA that had no tile).
struct TraceRec {
  uint32_t launch;               // sequence number of the launch since tracing began
  uint32_t cta;                  // blockIdx.x
  uint32_t kind;                 // ProductKind
  uint32_t tiles;                // tiles of the whole launch
  unsigned long long t_entry, t_mma_first, t_mma_last, t_exit;
  // leader's MMA thread, in SM cycles: from its start to the drain of its last
  // MMA, and within that the waits for operand stages to land and for an
  // accumulator to be freed by the epilogue
  unsigned long long mma_span_cycles, wait_operand_cycles, wait_accum_cycles;
};

// Launch arguments of the grouped Newton-Schulz product kernel.
//   symmetric product (m x m output, upper-triangle tiles, mirrored):
//     out = alpha * I + beta * aux + gamma * (L R^T)
//   full product (m x n output):
//     out = alpha * aux + gamma * (L R)        (L: m x m, R: m x n)
//     for a tall bucket the X slots hold Y = X^T, and the same launch computes
//     Y' = alpha * Y + gamma * (Y L) instead (L symmetric): sL names the m x m
//     operand and sR the X slot in both cases
// When `shift` is set, alpha becomes alpha + shift_sign * shift[matrix] per
// matrix (internal order).
struct GemmArgs {
  const Bucket* buckets;
  const unsigned char* tmaps;    // CUtensorMap array, 128 bytes each
  const int* sym_tiles;          // (ti << 16) | tj
  const InternalMat* imat;
  __nv_bfloat16* packed;
  int* err;
  int n_buckets;
  int total_tiles;
  int tile_base;                 // tile index of the launch's first tile (buckets[0]'s prefix)
  int sL, sR, sAux, sOut;
  const float* shift;            // per-matrix diagonal shift, or null
  int final_out;                 // full product: write O into `packed`
  float alpha, beta, gamma;
  float shift_sign;
  TraceRec* trace;               // this launch's records (gridDim.x of them), or null
  uint32_t trace_launch;
};

}  // namespace dm
