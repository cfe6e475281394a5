// C ABI of the owner-side Muon step: argument checks, planning, workspace
// layout, tensor maps, and the launch sequence.  See include/dmuon.h.
#include "dmuon.h"
#include "launch.h"
#include "tables.h"

#include <cuda.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <functional>
#include <cmath>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>
#include <vector>

namespace dm {
namespace {

constexpr size_t kHdrBytes = 256;  // workspace header: device error word
constexpr int kMaxNsSteps = 1000;
constexpr int kMaxDevices = 64;
constexpr float kDefaultAbc[3] = {3.4445f, -4.7750f, 2.0315f};
constexpr float kDefaultEps = 1e-7f;

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }
long long ceil_div(long long a, long long b) { return (a + b - 1) / b; }

// ------------------------------------------------------------------ planning
struct BucketPlan {
  int m = 0, n = 0;
  bool gram = false;
  bool tall = false;      // rows > cols: X slots hold Y = X^T (n x m), the parameter's layout
  std::vector<int> mats;  // caller indices, in caller order
  int pitch_x = 0, pitch_m = 0;
  long long stride_x = 0, stride_m = 0;
  bool used[kSlots] = {};
  size_t slot_off[kSlots] = {};
  std::vector<int> sym;   // (ti << 16) | tj, upper-triangle tiles of an m x m product
  int full_ti = 0, full_tj = 0;
  int first = 0;                    // table position of the first matrix
  long long chunk_lo = 0, chunks = 0;  // its elementwise chunks
  int sym_begin = 0, full_begin = 0;  // first product tile of the bucket within its group
};

struct Plan {
  int n = 0;
  std::vector<BucketPlan> buckets;  // standard buckets first, then Gram buckets
  int n_std = 0;                    // number of standard buckets
  std::vector<int> bucket_of, idx_in_bucket, internal_of;
  std::vector<long long> chunk_begin;              // per caller matrix
  std::vector<long long> partial_begin;            // per caller matrix, caller order
  std::vector<int> n_chunks;                       // per caller matrix
  std::vector<int> ew_order;                        // table position -> caller matrix
  std::vector<int> ew_pos;                          // caller matrix -> table position
  long long total_chunks = 0;
  int n_internal = 0;
  int sym_total = 0;
  size_t off_tables = 0, tables_bytes = 0;
  size_t off_ew = 0, off_bk = 0, off_imat = 0, off_sym = 0, off_tmaps = 0;
  size_t off_partials = 0, off_inv = 0, off_shift = 0;
  size_t prefix = 0;  // header, tables, norms: all that pack / update use; same for both variants
  size_t total = 0;
};

bool shape_ok(const dmuon_shape& s) {
  if (s.rows < 0 || s.cols < 0) return false;
  if (s.rows == 0 || s.cols == 0) return true;
  const int64_t m = std::min(s.rows, s.cols), n = std::max(s.rows, s.cols);
  return m <= DMUON_MAX_M && n <= DMUON_MAX_N;
}

// Accuracy rule of the Gram form with bf16 operands.  The Gram iteration
// works on A = X0 X0^T, whose eigenvalues are the squared singular values of
// X0: the closer to square a matrix is, the closer to zero its smallest
// singular values come, and squaring them loses them in bf16 rounding; very
// wide matrices lose accuracy too, and the rounding compounds with every step.
// So the form is used only inside a band of aspect ratios n/m that depends on
// the step count.  Each band is the measured one: over seeded Gaussian inputs
// with m = 256, 448 (both orientations) and 1024, aspect ratios 1.25 to 8, the
// worst relative error of the Gram result against the fp64 oracle stayed
// below 0.9 x the Newton-Schulz tolerance (2e-2 up to 5 steps, 4e-2 above)
// at every measured ratio from `lo` to `hi`.  Other step counts (0, 1 where
// Gram saves nothing, 11 and more, not measured) run the standard form.
struct GramBand {
  int steps;
  double lo, hi;  // Gram iff round(lo * m) <= n <= round(hi * m), as the measured shapes
};
constexpr GramBand kGramBand[] = {{2, 1.25, 8.0}, {3, 1.25, 8.0}, {4, 1.75, 8.0},
                                  {5, 1.75, 7.0}, {6, 1.25, 8.0}, {7, 1.5, 8.0},
                                  {8, 1.5, 8.0},  {9, 1.5, 7.0},  {10, 1.75, 5.83}};
constexpr int kGramMaxSteps = 10;

bool uses_gram(int variant, int m, int n, int ns_steps) {
  if (variant == DMUON_NS_GRAM_ALL) return n > m;
  if (variant != DMUON_NS_GRAM || n <= m) return false;
  for (const GramBand& b : kGramBand)
    if (b.steps == ns_steps)
      return n >= std::llround(b.lo * m) && n <= std::llround(b.hi * m);
  return false;
}

bool variant_ok(int variant) {
  return variant == DMUON_NS_STANDARD || variant == DMUON_NS_GRAM ||
         variant == DMUON_NS_GRAM_ALL;
}

int build_plan(int n, const dmuon_shape* shp, int variant, int ns_steps, Plan& P) {
  if (n < 0 || (n > 0 && shp == nullptr)) return DMUON_ERR_INVALID_ARG;
  if (!variant_ok(variant)) return DMUON_ERR_INVALID_ARG;
  P = Plan();
  P.n = n;
  P.bucket_of.assign(n, -1);
  P.idx_in_bucket.assign(n, -1);
  P.internal_of.assign(n, -1);
  P.chunk_begin.assign(n, 0);
  P.partial_begin.assign(n, 0);
  P.n_chunks.assign(n, 0);

  // buckets keyed by (gram, m, n, tall); standard first, each group in
  // first-seen order
  using Key = std::tuple<int, int, int, int>;
  std::map<Key, int> key_to_b;
  std::vector<Key> order;
  for (int i = 0; i < n; ++i) {
    if (!shape_ok(shp[i])) return DMUON_ERR_INVALID_ARG;
    const long long r = shp[i].rows, c = shp[i].cols;
    P.n_chunks[i] = int(ceil_div(r * c, kChunk));
    if (r == 0 || c == 0) continue;
    const int m = int(std::min(r, c)), nn = int(std::max(r, c));
    const Key key(uses_gram(variant, m, nn, ns_steps) ? 1 : 0, m, nn, r > c ? 1 : 0);
    if (!key_to_b.count(key)) {
      key_to_b[key] = -1;
      order.push_back(key);
    }
  }
  // within each group, wide/square buckets before tall ones, so that every
  // product launch splits into few runs of one orientation
  std::stable_sort(order.begin(), order.end(), [](const Key& a, const Key& b) {
    return std::make_pair(std::get<0>(a), std::get<3>(a)) <
           std::make_pair(std::get<0>(b), std::get<3>(b));
  });
  for (size_t b = 0; b < order.size(); ++b) {
    key_to_b[order[b]] = int(b);
    BucketPlan bp;
    bp.gram = std::get<0>(order[b]) != 0;
    bp.m = std::get<1>(order[b]);
    bp.n = std::get<2>(order[b]);
    bp.tall = std::get<3>(order[b]) != 0;
    P.buckets.push_back(bp);
    if (!bp.gram) P.n_std = int(b) + 1;
  }
  for (int i = 0; i < n; ++i) {
    const long long r = shp[i].rows, c = shp[i].cols;
    if (r == 0 || c == 0) continue;
    const int m = int(std::min(r, c)), nn = int(std::max(r, c));
    const int b = key_to_b[Key(uses_gram(variant, m, nn, ns_steps) ? 1 : 0, m, nn, r > c ? 1 : 0)];
    P.bucket_of[i] = b;
    P.idx_in_bucket[i] = int(P.buckets[b].mats.size());
    P.buckets[b].mats.push_back(i);
  }
  int internal = 0;
  for (auto& B : P.buckets) {
    for (int i : B.mats) P.internal_of[i] = internal++;
    // X slots in the parameter's orientation: m x n, or n x m for a tall bucket
    const int x_rows = B.tall ? B.n : B.m, x_cols = B.tall ? B.m : B.n;
    B.pitch_x = int(align_up(size_t(x_cols), 64));
    B.pitch_m = int(align_up(size_t(B.m), 64));
    B.stride_x = (long long)x_rows * B.pitch_x;
    B.stride_m = (long long)B.m * B.pitch_m;
    if (!B.gram) {
      B.used[SX0] = B.used[SX1] = B.used[SM0] = B.used[SM1] = true;
    } else {
      B.used[SX0] = true;
      for (int s = SM0; s <= SM5; ++s) B.used[s] = true;
    }
    // upper-triangle 256 x 256 tiles (diagonal tiles included) of an m x m product
    const int J = int(ceil_div(B.m, kTileM));
    for (int ti = 0; ti < J; ++ti)
      for (int tj = ti; tj < J; ++tj) B.sym.push_back((ti << 16) | tj);
    // tile grid of the m x n product's output (X' or Y')
    B.full_ti = int(ceil_div(x_rows, kTileM));
    B.full_tj = int(ceil_div(x_cols, kTileN));
    P.sym_total += int(B.sym.size());
  }
  P.n_internal = internal;

  // The per-matrix table follows the internal (bucket-major) order, empty
  // matrices last, so that every bucket -- and every run of buckets -- is one
  // contiguous range of table entries and elementwise chunks.
  P.ew_pos.assign(n, -1);
  for (const auto& B : P.buckets)
    for (int i : B.mats) P.ew_order.push_back(i);
  for (int i = 0; i < n; ++i)
    if (P.bucket_of[i] < 0) P.ew_order.push_back(i);
  long long partials = 0;
  for (int i = 0; i < n; ++i) {
    P.partial_begin[i] = partials;
    partials += P.n_chunks[i];
  }
  for (int k = 0; k < n; ++k) {
    const int i = P.ew_order[k];
    P.ew_pos[i] = k;
    P.chunk_begin[i] = P.total_chunks;
    P.total_chunks += P.n_chunks[i];
  }
  // product tile numbering: one sequence over the standard buckets, another
  // over the Gram buckets (each group's launches start at its first bucket)
  long long sym_begin = 0, full_begin = 0;
  for (size_t b = 0; b < P.buckets.size(); ++b) {
    BucketPlan& B = P.buckets[b];
    if (int(b) == P.n_std) sym_begin = full_begin = 0;
    B.first = P.ew_pos[B.mats.front()];
    B.chunk_lo = P.chunk_begin[B.mats.front()];
    for (int i : B.mats) B.chunks += P.n_chunks[i];
    B.sym_begin = int(sym_begin);
    B.full_begin = int(full_begin);
    sym_begin += (long long)B.mats.size() * (long long)B.sym.size();
    full_begin += (long long)B.mats.size() * B.full_ti * B.full_tj;
    if (sym_begin > INT32_MAX || full_begin > INT32_MAX) return DMUON_ERR_UNSUPPORTED;
  }

  // workspace layout
  size_t off = kHdrBytes;
  P.off_tables = off;
  P.off_ew = off;
  off = align_up(off + size_t(n) * sizeof(EwMat), 16);
  P.off_bk = off;
  off = align_up(off + P.buckets.size() * sizeof(Bucket), 16);
  P.off_imat = off;
  off = align_up(off + size_t(P.n_internal) * sizeof(InternalMat), 16);
  P.off_sym = off;
  off = align_up(off + size_t(P.sym_total) * sizeof(int), 16);
  // the TMA unit reads a tensor map only from a 64-byte aligned address
  off = align_up(off, 128);
  P.off_tmaps = off;
  off = align_up(off + P.buckets.size() * kMapsPerBucket * 128, 16);
  P.tables_bytes = off - P.off_tables;
  off = align_up(off, 256);
  P.off_partials = off;
  off = align_up(off + size_t(P.total_chunks) * sizeof(float), 256);
  P.off_inv = off;
  off = align_up(off + size_t(n) * sizeof(float), 256);
  P.off_shift = off;
  off = align_up(off + size_t(P.n_internal) * sizeof(float), 4096);
  P.prefix = off;
  for (auto& B : P.buckets) {
    for (int s = 0; s < kSlots; ++s) {
      if (!B.used[s]) continue;
      B.slot_off[s] = off;
      const long long stride = slot_is_x(s) ? B.stride_x : B.stride_m;
      off = align_up(off + size_t(B.mats.size()) * size_t(stride) * 2, 4096);
    }
  }
  P.total = off;
  return DMUON_OK;
}

// ------------------------------------------------------------------ device
struct DevInfo {
  bool ready = false;
  int status = DMUON_OK;
  int sms = 0;
  int clock_khz = 0;
  int max_clusters = 0;  // resident CTA pairs of the product kernel
  // Lowest-priority stream on which a whole step runs its memory-bound kernels
  // next to the products (null: the step runs on the caller's stream alone).
  // This one serves callers whose stream is being captured and callers beyond
  // the per-stream table below.
  cudaStream_t aux = nullptr;
};
std::mutex g_mu;
DevInfo g_dev[kMaxDevices];

// Each caller stream gets its own lowest-priority companion stream (up to
// kAuxPerDevice caller streams per device), so that owners stepping on
// different caller streams do not queue behind each other's memory-bound work.
// Past that many streams, or while the caller's stream is being captured into
// a graph (no stream is created then), the device's shared companion serves;
// sharing it serialises that work but never changes a result, since every
// piece of it is ordered against its own caller stream by events.
constexpr int kAuxPerDevice = 16;
struct AuxEntry {
  cudaStream_t caller = nullptr;
  cudaStream_t aux = nullptr;
};
AuxEntry g_aux[kMaxDevices][kAuxPerDevice];
int g_aux_used[kMaxDevices] = {};

int device_info(DevInfo* out) {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return DMUON_ERR_CUDA;
  if (d < 0 || d >= kMaxDevices) return DMUON_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lk(g_mu);
  DevInfo& D = g_dev[d];
  if (!D.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&D.sms, cudaDevAttrMultiProcessorCount, d) != cudaSuccess ||
        cudaDeviceGetAttribute(&D.clock_khz, cudaDevAttrClockRate, d) != cudaSuccess)
      return DMUON_ERR_CUDA;
    if (major != 10 || minor != 3) {
      D.status = DMUON_ERR_UNSUPPORTED;
    } else if (ns_gemm_prepare(D.sms, &D.max_clusters) != cudaSuccess) {
      return DMUON_ERR_CUDA;
    } else {
      int least = 0, greatest = 0;
      if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
          cudaStreamCreateWithPriority(&D.aux, cudaStreamNonBlocking, least) != cudaSuccess) {
        D.aux = nullptr;
        (void)cudaGetLastError();
      }
    }
    D.ready = true;
  }
  *out = D;
  return D.status;
}

// Companion stream of `caller` on the current device (D from device_info).
cudaStream_t aux_stream_for(const DevInfo& D, cudaStream_t caller) {
  if (D.aux == nullptr) return nullptr;
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return D.aux;
  std::lock_guard<std::mutex> lk(g_mu);
  for (int k = 0; k < g_aux_used[d]; ++k)
    if (g_aux[d][k].caller == caller) return g_aux[d][k].aux;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if (cudaStreamIsCapturing(caller, &cap) != cudaSuccess || cap != cudaStreamCaptureStatusNone) {
    (void)cudaGetLastError();
    return D.aux;
  }
  if (g_aux_used[d] >= kAuxPerDevice) return D.aux;
  int least = 0, greatest = 0;
  cudaStream_t x = nullptr;
  if (cudaDeviceGetStreamPriorityRange(&least, &greatest) != cudaSuccess ||
      cudaStreamCreateWithPriority(&x, cudaStreamNonBlocking, least) != cudaSuccess) {
    (void)cudaGetLastError();
    return D.aux;
  }
  g_aux[d][g_aux_used[d]].caller = caller;
  g_aux[d][g_aux_used[d]].aux = x;
  ++g_aux_used[d];
  return x;
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// One 3-D map (cols, rows, matrix) over a slot.  Operand maps move 64 x 64
// boxes with the 128-byte swizzle that the MMA descriptors expect; epilogue
// maps move the 32 x 32 chunks of one epilogue warp with the 64-byte swizzle
// (one 64-byte row per chunk row).  Reads outside (cols, rows) are zero-filled
// and writes outside are dropped, which handles ragged edges.
bool encode_slot_map(CUtensorMap* map, void* base, int cols, int rows, int count, int pitch,
                     long long stride, bool epilogue) {
  auto enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  const cuuint64_t dims[3] = {cuuint64_t(cols), cuuint64_t(rows), cuuint64_t(count)};
  const cuuint64_t strides[2] = {cuuint64_t(pitch) * 2, cuuint64_t(stride) * 2};
  const cuuint32_t box_op[3] = {64, 64, 1};
  const cuuint32_t box_epi[3] = {32, 32, 1};
  const cuuint32_t es[3] = {1, 1, 1};
  return enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, base, dims, strides,
             epilogue ? box_epi : box_op, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
             epilogue ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B,
             CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ------------------------------------------------------------------ one call
struct Request {
  int n = 0;
  const dmuon_shape* shp = nullptr;
  const void* const* grad = nullptr;
  int grad_dt = DMUON_BF16;
  float* const* momentum = nullptr;
  void* const* weight = nullptr;
  int weight_dt = DMUON_BF16;
  const int64_t* offset = nullptr;
  void* packed = nullptr;
  void* ws = nullptr;
  size_t ws_bytes = 0;
  int variant = DMUON_NS_STANDARD;
  cudaStream_t stream = nullptr;
  bool do_pack = false, do_ns = false, do_update = false;
  float beta = 0.95f;
  int ns_steps = 5;
  float abc[3] = {kDefaultAbc[0], kDefaultAbc[1], kDefaultAbc[2]};
  float eps = kDefaultEps;
  bool pack_norms = false;
  float lr = 0.02f;
};

int check_request(const Request& R, const Plan& P) {
  if (R.packed == nullptr || R.ws == nullptr || R.offset == nullptr) return DMUON_ERR_INVALID_ARG;
  if (!aligned(R.packed, 256) || !aligned(R.ws, 256)) return DMUON_ERR_ALIGNMENT;
  // pack and update never touch the Newton-Schulz buffers; their part of the
  // layout does not depend on the variant
  if (R.ws_bytes < (R.do_ns ? P.total : P.prefix)) return DMUON_ERR_WORKSPACE;
  if (R.do_pack) {
    if (R.grad == nullptr || R.momentum == nullptr) return DMUON_ERR_INVALID_ARG;
    if (R.grad_dt != DMUON_F32 && R.grad_dt != DMUON_BF16) return DMUON_ERR_INVALID_ARG;
    if (!std::isfinite(R.beta)) return DMUON_ERR_INVALID_ARG;
  }
  if (R.do_update) {
    if (R.weight == nullptr) return DMUON_ERR_INVALID_ARG;
    if (R.weight_dt != DMUON_F32 && R.weight_dt != DMUON_BF16) return DMUON_ERR_INVALID_ARG;
    if (!std::isfinite(R.lr)) return DMUON_ERR_INVALID_ARG;
  }
  if (R.do_ns) {
    if (R.ns_steps < 0 || R.ns_steps > kMaxNsSteps) return DMUON_ERR_INVALID_ARG;
    if (!(R.eps >= 0.f) || !std::isfinite(R.eps)) return DMUON_ERR_INVALID_ARG;
    for (float v : R.abc)
      if (!std::isfinite(v)) return DMUON_ERR_INVALID_ARG;
  }
  for (int i = 0; i < R.n; ++i) {
    const bool active = R.shp[i].rows > 0 && R.shp[i].cols > 0;
    if (!active) continue;
    if (R.offset[i] < 0 || R.offset[i] % DMUON_PACK_ALIGN_ELEMS != 0) return DMUON_ERR_ALIGNMENT;
    if (R.do_pack && (R.grad[i] == nullptr || R.momentum[i] == nullptr))
      return DMUON_ERR_INVALID_ARG;
    if (R.do_update && R.weight[i] == nullptr) return DMUON_ERR_INVALID_ARG;
  }
  return DMUON_OK;
}

int upload_tables(const Request& R, const Plan& P) {
  std::vector<unsigned char> blob(P.tables_bytes, 0);
  unsigned char* ws = static_cast<unsigned char*>(R.ws);
  auto at = [&](size_t off) { return blob.data() + (off - P.off_tables); };
  EwMat* ew = reinterpret_cast<EwMat*>(at(P.off_ew));
  Bucket* bk = reinterpret_cast<Bucket*>(at(P.off_bk));
  InternalMat* im = reinterpret_cast<InternalMat*>(at(P.off_imat));
  int* sym = reinterpret_cast<int*>(at(P.off_sym));
  CUtensorMap* maps = reinterpret_cast<CUtensorMap*>(at(P.off_tmaps));
  // a tensor map the TMA unit cannot read faults the kernel: refuse instead
  if ((reinterpret_cast<uintptr_t>(ws + P.off_tmaps) & 63u) != 0) return DMUON_ERR_ALIGNMENT;

  for (int i = 0; i < P.n; ++i) {
    EwMat& E = ew[P.ew_pos[i]];
    const long long r = R.shp[i].rows, c = R.shp[i].cols;
    E.rows = int(r);
    E.cols = int(c);
    E.numel = r * c;
    E.active = (r > 0 && c > 0) ? 1 : 0;
    E.chunk_begin = P.chunk_begin[i];
    E.partial_begin = P.partial_begin[i];
    E.n_chunks = P.n_chunks[i];
    E.packed_off = E.active ? R.offset[i] : 0;
    E.upd_scale = float(std::sqrt(std::max(1.0, double(r) / double(std::max<long long>(c, 1)))));
    if (R.do_pack && E.active) {
      E.g = R.grad[i];
      E.mom = R.momentum[i];
      if (aligned(E.g, 16) && aligned(E.mom, 16)) E.flags |= kFlagVecGM;
    }
    if (R.do_update && E.active) {
      E.w = R.weight[i];
      if (aligned(E.w, 16)) E.flags |= kFlagVecW;
    }
    if (c % 8 == 0) E.flags |= kFlagRowsAligned;
    const int b = P.bucket_of[i];
    if (b >= 0) {
      const BucketPlan& B = P.buckets[b];
      E.pitch_x = B.pitch_x;
      E.x0 = reinterpret_cast<__nv_bfloat16*>(ws + B.slot_off[SX0]) +
             (long long)P.idx_in_bucket[i] * B.stride_x;
      InternalMat& M = im[P.internal_of[i]];
      M.packed_off = R.offset[i];
      M.caller = i;
    }
  }
  int sym_off = 0, internal = 0;
  for (size_t b = 0; b < P.buckets.size(); ++b) {
    const BucketPlan& BP = P.buckets[b];
    Bucket& B = bk[b];
    B.m = BP.m;
    B.n = BP.n;
    B.count = int(BP.mats.size());
    B.first = internal;
    internal += B.count;
    B.pitch_x = BP.pitch_x;
    B.pitch_m = BP.pitch_m;
    B.stride_x = BP.stride_x;
    B.stride_m = BP.stride_m;
    B.tall = BP.tall ? 1 : 0;
    B.tmap = int(b) * kMapsPerBucket;
    for (int s = 0; s < kSlots; ++s) {
      if (!BP.used[s] || !R.do_ns) continue;
      void* base = ws + BP.slot_off[s];
      B.slot[s] = static_cast<__nv_bfloat16*>(base);
      const bool x = slot_is_x(s);
      const int cols = x && !BP.tall ? BP.n : BP.m, rows = x && BP.tall ? BP.n : BP.m;
      for (int epi = 0; epi < 2; ++epi)
        if (!encode_slot_map(&maps[b * kMapsPerBucket + epi * kSlots + s], base, cols, rows,
                             B.count, x ? BP.pitch_x : BP.pitch_m,
                             x ? BP.stride_x : BP.stride_m, epi != 0))
          return DMUON_ERR_CUDA;
    }
    B.sym_off = sym_off;
    B.sym_count = int(BP.sym.size());
    std::memcpy(sym + sym_off, BP.sym.data(), BP.sym.size() * sizeof(int));
    sym_off += B.sym_count;
    B.full_ti = BP.full_ti;
    B.full_tj = BP.full_tj;
    B.sym_begin = BP.sym_begin;
    B.full_begin = BP.full_begin;
  }
  if (launch_upload(ws + P.off_tables, blob.data(), blob.size(), R.stream) != cudaSuccess)
    return DMUON_ERR_CUDA;
  return DMUON_OK;
}

// One run of Newton-Schulz product launches over the buckets [b0, b1) of one
// group (standard or Gram), on `stream`.
struct GemmLauncher {
  const Plan& P;
  const Request& R;
  int clusters;
  unsigned char* ws;
  int b0, b1;
  cudaStream_t stream;

  GemmLauncher(const Plan& p, const Request& r, int c, unsigned char* w, int lo, int hi,
               cudaStream_t s)
      : P(p), R(r), clusters(c), ws(w), b0(lo), b1(hi), stream(s) {}
  GemmArgs base() const {
    GemmArgs g{};
    g.buckets = reinterpret_cast<const Bucket*>(ws + P.off_bk) + b0;
    g.tmaps = ws + P.off_tmaps;
    g.sym_tiles = reinterpret_cast<const int*>(ws + P.off_sym);
    g.imat = reinterpret_cast<const InternalMat*>(ws + P.off_imat);
    g.packed = static_cast<__nv_bfloat16*>(R.packed);
    g.err = reinterpret_cast<int*>(ws);
    g.n_buckets = b1 - b0;
    return g;
  }
  // One launch per run of consecutive buckets that need the same product kind
  // (the planner keeps buckets of one orientation together within a group).
  bool launch_runs(GemmArgs g, bool full, bool by_orientation) const {
    int b = b0;
    while (b < b1) {
      const bool tall = P.buckets[b].tall;
      int e = b + 1;
      long long tiles = 0;
      if (by_orientation)
        while (e < b1 && P.buckets[e].tall == tall) ++e;
      else
        e = b1;
      for (int k = b; k < e; ++k) {
        const BucketPlan& B = P.buckets[k];
        tiles += (long long)B.mats.size() * (full ? (long long)B.full_ti * B.full_tj
                                                  : (long long)B.sym.size());
      }
      g.buckets = reinterpret_cast<const Bucket*>(ws + P.off_bk) + b;
      g.n_buckets = e - b;
      g.tile_base = full ? P.buckets[b].full_begin : P.buckets[b].sym_begin;
      g.total_tiles = int(tiles);
      const int kind = full ? (tall ? kFullTall : kFullWide)
                            : (by_orientation && tall ? kSymMN : kSymK);
      if (launch_ns_gemm(g, kind, clusters, stream) != cudaSuccess) return false;
      b = e;
    }
    return true;
  }
  // out = alpha*I + beta*aux + gamma*L R^T  (m x m, symmetric)
  bool sym(int sL, int sR, int sAux, int sOut, float alpha, float beta, float gamma,
           const float* shift = nullptr, float shift_sign = 0.f) const {
    GemmArgs g = base();
    g.sL = sL; g.sR = sR; g.sAux = sAux; g.sOut = sOut;
    g.alpha = alpha; g.beta = beta; g.gamma = gamma;
    g.shift = shift; g.shift_sign = shift_sign;
    // X X^T reads the X slots, whose layout follows the orientation
    return launch_runs(g, false, slot_is_x(sL));
  }
  // out = alpha*aux + gamma*L R  (m x n; Y' = alpha*Y + gamma*Y L for tall
  // buckets); final: write O into the packed buffer
  bool full(int sL, int sR, int sAux, int sOut, float alpha, float gamma, bool final,
            const float* shift = nullptr, float shift_sign = 0.f) const {
    GemmArgs g = base();
    g.sL = sL; g.sR = sR; g.sAux = sAux; g.sOut = sOut;
    g.alpha = alpha; g.beta = 0.f; g.gamma = gamma;
    g.shift = shift; g.shift_sign = shift_sign;
    g.final_out = final ? 1 : 0;
    return launch_runs(g, true, true);
  }
  int first() const { return P.buckets[b0].first; }
  int n_mats() const {
    int k = 0;
    for (int b = b0; b < b1; ++b) k += int(P.buckets[b].mats.size());
    return k;
  }
};

// Standard Newton-Schulz on buckets [b0, b1), per step:
//   A = X X^T;  d = b s + c s^2 with s = trace(A)/m;
//   B' = b A + c A A - d I;  X' = (a + d) X + B' X   (= a X + B X)
// Storing B' instead of B keeps B's large diagonal (about b + c once the
// singular values approach 1) out of the bf16 rounding, where it would be
// amplified by the cancellation between a X and B X.
// `before(i)`, when given, runs before product launch i = 3*step + {0: X X^T,
// 1: A A, 2: B X} is enqueued.
bool ns_standard(const GemmLauncher& L, const Request& R, const Plan& P, unsigned char* ws,
                 const std::function<bool(int)>& before = nullptr) {
  const float a = R.abc[0], b = R.abc[1], c = R.abc[2];
  float* shift = reinterpret_cast<float*>(ws + P.off_shift);
  const Bucket* bk = reinterpret_cast<const Bucket*>(ws + P.off_bk) + L.b0;
  auto hook = [&](int i) { return !before || before(i); };
  for (int k = 0; k < R.ns_steps; ++k) {
    const int xin = (k & 1) ? SX1 : SX0, xout = (k & 1) ? SX0 : SX1;
    const bool last = k + 1 == R.ns_steps;
    if (!hook(3 * k) || !L.sym(xin, xin, SM0, SM0, 0.f, 0.f, 1.f)) return false;
    if (launch_diag_shift(bk, L.b1 - L.b0, L.first(), L.n_mats(), SM0, b, c, shift, L.stream) !=
        cudaSuccess)
      return false;
    if (!hook(3 * k + 1) || !L.sym(SM0, SM0, SM0, SM1, 0.f, b, c, shift, -1.f)) return false;
    if (!hook(3 * k + 2) || !L.full(SM1, xin, xin, xout, a, 1.f, last, shift, 1.f)) return false;
  }
  return true;
}

// Gram Newton-Schulz on buckets [b0, b1): A0 = X0 X0^T; per step
// P = aI + bA + cA^2, Q = P Q, A' = A P^2; finally O = Q X0.  Slots: A in
// SM0/SM1, P in SM2 (SM3 at step 0, where Q = P), Q in SM3/SM4, T = P^2 in SM5.
// `before(i)`, when given, runs before the i-th product launch is enqueued
// (the order of gram_launches below).
bool ns_gram(const GemmLauncher& L, const Request& R,
             const std::function<bool(int)>& before = nullptr) {
  const float a = R.abc[0], b = R.abc[1], c = R.abc[2];
  int i = 0;
  auto hook = [&]() { return !before || before(i++); };
  int sA = SM0, sAn = SM1, sQ = SM3, sQn = SM4;
  if (!hook() || !L.sym(SX0, SX0, SM0, sA, 0.f, 0.f, 1.f)) return false;
  for (int k = 0; k < R.ns_steps; ++k) {
    const bool last = k + 1 == R.ns_steps;
    const int sP = (k == 0) ? SM3 : SM2;
    if (!hook() || !L.sym(sA, sA, sA, sP, a, b, c)) return false;
    if (k > 0) {
      if (!hook() || !L.sym(sP, sQ, SM0, sQn, 0.f, 0.f, 1.f)) return false;
      std::swap(sQ, sQn);
    }
    if (!last) {
      if (!hook() || !L.sym(sP, sP, SM0, SM5, 0.f, 0.f, 1.f)) return false;
      if (!hook() || !L.sym(sA, SM5, SM0, sAn, 0.f, 0.f, 1.f)) return false;
      std::swap(sA, sAn);
    }
  }
  return hook() && L.full(sQ, SX0, SX0, SX0, 0.f, 1.f, true);
}

// The product launches of one Newton-Schulz run over a group of buckets, in
// issue order, as the time model needs them: full (m x n output) or
// symmetric (m x m), and whether the reduction runs over n (X X^T) or m.
struct ProductLaunch {
  bool full, k_is_n;
};

std::vector<ProductLaunch> standard_launches(int ns_steps) {
  std::vector<ProductLaunch> v;
  for (int k = 0; k < ns_steps; ++k) {
    v.push_back({false, true});   // X X^T
    v.push_back({false, false});  // A A
    v.push_back({true, false});   // B X
  }
  return v;
}

std::vector<ProductLaunch> gram_launches(int ns_steps) {
  std::vector<ProductLaunch> v;
  v.push_back({false, true});     // X0 X0^T
  for (int k = 0; k < ns_steps; ++k) {
    v.push_back({false, false});  // P
    if (k > 0) v.push_back({false, false});           // P Q
    if (k + 1 < ns_steps) {
      v.push_back({false, false});  // P P
      v.push_back({false, false});  // A P^2
    }
  }
  v.push_back({true, false});     // Q X0
  return v;
}

// ------------------------------------------------------------------ step pipeline
// The whole step runs its buckets in positions -- a position is a run
// of buckets (consecutive in the plan) whose products share launches -- and
// overlaps its memory-bound work (momentum + pack, norm finish and relayout of
// later positions; weight update of earlier ones) with the tensor-core
// products of the current position, on a second, low-priority stream.  That
// work is enqueued in pieces, each one gated to start together with one long
// product launch and sized to finish inside it: a product launch ready to
// start while a memory-bound grid still has blocks pending waits until that
// whole grid is dispatched (an SM filled with memory-bound blocks has no room
// for a product CTA, about 38k registers, and the block scheduler keeps
// refilling it from the pending grid), whereas memory-bound blocks enqueued
// next to a resident product launch run in the room its CTAs leave and never
// hold up the next launch.  What cannot be placed runs on the caller's stream
// at full speed: the packs of the first positions before any product, the
// last position's update after all of them.
//
// Time model (for choosing and sizing, not for results): a product launch
// takes its busiest CTA pair's share of tile work (tiles go round-robin to the
// pairs) at kModelPairFlops, plus kModelLaunchSeconds; memory-bound work moves
// kModelHbmBytes alone and kModelCoBytes next to a product launch, of which a
// piece may plan to use kSlotFill.
constexpr double kModelPairFlops = 2.2e13;
constexpr double kModelLaunchSeconds = 2e-5;
constexpr double kModelHbmBytes = 6.5e12;
constexpr double kModelCoBytes = 3.0e12;
constexpr double kSlotFill = 0.45;
constexpr double kMinPieceBytes = 64.0 * (1 << 20);

enum PieceKind : int { kPiecePack = 0, kPieceFinalize = 1, kPieceRelayout = 2, kPieceUpdate = 3 };
struct Piece {
  int kind = 0, bucket = 0;
  long long lo = 0, hi = 0;  // chunk range within the bucket
};

struct StepSchedule {
  std::vector<std::pair<int, int>> pos;               // bucket range [b0, b1) of each position
  std::vector<std::vector<Piece>> pre;               // per position: its pack work left for `s`,
                                                      // right before its products
  std::vector<std::vector<std::vector<Piece>>> slot;  // [position][launch]: pieces next to it
  std::vector<Piece> tail_update;                     // update ranges run on `s` at the end
  double products = 0.0, exposed = 0.0;               // modelled seconds
};

// Modelled seconds of one product over the buckets [b0, b1): one launch per
// run of buckets of one orientation, as the launcher issues them.
double model_product_seconds(const Plan& P, int b0, int b1, const ProductLaunch& pl,
                             int clusters) {
  const int phase = pl.full ? 2 : 1;
  double total = 0.0;
  std::vector<double> load;
  int b = b0;
  while (b < b1) {
    int e = b + 1;
    while (e < b1 && P.buckets[e].tall == P.buckets[b].tall) ++e;
    long long tiles = 0;
    for (int k = b; k < e; ++k) {
      const BucketPlan& B = P.buckets[k];
      tiles += (long long)B.mats.size() *
               (phase == 2 ? (long long)B.full_ti * B.full_tj : (long long)B.sym.size());
    }
    const int C = int(std::min<long long>(tiles, clusters));
    if (C > 0) {
      load.assign(size_t(C), 0.0);
      long long first = 0;
      for (int k = b; k < e; ++k) {
        const BucketPlan& B = P.buckets[k];
        const long long n = (long long)B.mats.size() *
                            (phase == 2 ? (long long)B.full_ti * B.full_tj : (long long)B.sym.size());
        const double K = pl.k_is_n ? double(B.n) : double(B.m);
        const double cost = 2.0 * kTileM * kTileN * K;
        const long long q = n / C, rem = n % C;
        for (int c = 0; c < C; ++c) load[size_t(c)] += double(q) * cost;
        for (long long r = 0; r < rem; ++r) load[size_t((first + r) % C)] += cost;
        first += n;
      }
      total += *std::max_element(load.begin(), load.end()) / kModelPairFlops + kModelLaunchSeconds;
    }
    b = e;
  }
  return total;
}

struct PieceCosts {
  double pack_chunk, relay_chunk, update_chunk;  // bytes moved per chunk
};

PieceCosts piece_costs(const Request& R) {
  const double g = R.grad_dt == DMUON_BF16 ? 2.0 : 4.0, w = R.weight_dt == DMUON_BF16 ? 2.0 : 4.0;
  return {double(kChunk) * (g + 4.0 + 4.0 + 2.0), double(kChunk) * 4.0,
          double(kChunk) * (2.0 + 2.0 * w)};
}

// Greedy placement for one sequence of positions.  Slots are the product
// phases in issue order; each takes, up to its budget, first the pack/relayout
// work of the nearest later position (needed before that position's products
// start), then the updates of earlier positions.  The part of a position's pack
// that the slots before it cannot take (all of it for the first position) runs
// on `s` just before its products, after the part that did run beside them.
StepSchedule plan_step(const Plan& P, const Request& R,
                       const std::vector<std::pair<int, int>>& pos, int clusters) {
  const int g = int(pos.size());
  const PieceCosts pc = piece_costs(R);
  StepSchedule S;
  S.pos = pos;
  S.pre.assign(size_t(g), {});
  std::vector<std::vector<double>> dur(static_cast<size_t>(g));
  S.products = 0.0;
  for (int k = 0; k < g; ++k) {
    const int b0 = pos[size_t(k)].first, b1 = pos[size_t(k)].second;
    const auto launches = P.buckets[b0].gram ? gram_launches(R.ns_steps)
                                             : standard_launches(R.ns_steps);
    for (const ProductLaunch& pl : launches) {
      dur[size_t(k)].push_back(model_product_seconds(P, b0, b1, pl, clusters));
      S.products += dur[size_t(k)].back();
    }
  }
  S.slot.assign(size_t(g), std::vector<std::vector<Piece>>());
  for (int k = 0; k < g; ++k) S.slot[size_t(k)].assign(dur[size_t(k)].size(), {});
  struct Todo { int pos, kind, bucket; long long lo, hi; };
  std::vector<Todo> mb, upd;
  for (int k = 0; k < g; ++k)
    for (int b = pos[size_t(k)].first; b < pos[size_t(k)].second; ++b) {
      const long long ch = P.buckets[b].chunks;
      mb.push_back({k, kPiecePack, b, 0, ch});
      mb.push_back({k, kPieceFinalize, b, 0, 1});
      mb.push_back({k, kPieceRelayout, b, 0, ch});
      upd.push_back({k, kPieceUpdate, b, 0, ch});
    }
  size_t mi = 0, ui = 0;
  for (int k = 0; k < g; ++k) {
    // a position's pack must be done before its products start: what the
    // earlier slots could not take runs on `s` just before them
    for (; mi < mb.size() && mb[mi].pos <= k; ++mi)
      if (mb[mi].lo < mb[mi].hi)
        S.pre[size_t(k)].push_back({mb[mi].kind, mb[mi].bucket, mb[mi].lo, mb[mi].hi});
    for (size_t i = 0; i < dur[size_t(k)].size(); ++i) {
      double budget = dur[size_t(k)][i] * kModelCoBytes * kSlotFill;
      if (budget < kMinPieceBytes) continue;
      std::vector<Piece>& out = S.slot[size_t(k)][i];
      auto take = [&](Todo& t, double unit_bytes) {
        const long long can = unit_bytes > 0 ? (long long)(budget / unit_bytes) : t.hi - t.lo;
        const long long n = std::min(can, t.hi - t.lo);
        if (n <= 0) return false;
        out.push_back({t.kind, t.bucket, t.lo, t.lo + n});
        budget -= double(n) * unit_bytes;
        t.lo += n;
        return t.lo == t.hi;
      };
      while (mi < mb.size()) {
        Todo& t = mb[mi];
        const double ub = t.kind == kPiecePack ? pc.pack_chunk
                          : t.kind == kPieceRelayout ? pc.relay_chunk : 0.0;
        if (!take(t, ub)) break;
        ++mi;
      }
      while (ui < upd.size() && upd[ui].pos < k) {
        if (!take(upd[ui], pc.update_chunk)) break;
        ++ui;
      }
    }
  }
  // updates left over (the unplaced rest of each) run on `s` after the last products
  S.tail_update.clear();
  for (; ui < upd.size(); ++ui)
    if (upd[ui].lo < upd[ui].hi)
      S.tail_update.push_back({kPieceUpdate, upd[ui].bucket, upd[ui].lo, upd[ui].hi});
  S.exposed = 0.0;
  for (const auto& v : S.pre)
    for (const Piece& t : v)
      S.exposed += double(t.hi - t.lo) *
                   (t.kind == kPiecePack ? pc.pack_chunk
                    : t.kind == kPieceRelayout ? pc.relay_chunk : 0.0) / kModelHbmBytes;
  for (const Piece& t : S.tail_update)
    S.exposed += double(t.hi - t.lo) * pc.update_chunk / kModelHbmBytes;
  return S;
}

// The candidate schedules of a whole step: one position per bucket, by size
// (short first products, small up-front packs), the same with the second
// position moved last (the last position's update is exposed), buckets too
// small to occupy every CTA pair joined with a neighbour, and one position per
// run of buckets with the same form and orientation (fewer, fuller launches for
// sets of small matrices).  The one with the least
// modelled product plus exposed time runs.  A position never mixes the
// standard and the Gram form.
StepSchedule choose_step_schedule(const Plan& P, const Request& R, int clusters) {
  const int nb = int(P.buckets.size());
  std::vector<int> ord(static_cast<size_t>(nb));
  for (int b = 0; b < nb; ++b) ord[size_t(b)] = b;
  std::stable_sort(ord.begin(), ord.end(), [&](int a, int b) {
    return P.buckets[a].chunks < P.buckets[b].chunks;
  });
  std::vector<std::vector<std::pair<int, int>>> cands;
  std::vector<std::pair<int, int>> one;
  for (int b : ord) one.push_back({b, b + 1});
  cands.push_back(one);
  if (nb >= 3) {
    std::vector<std::pair<int, int>> alt = one;
    const auto second = alt[1];
    alt.erase(alt.begin() + 1);
    alt.push_back(second);
    cands.push_back(alt);
  }
  auto chunks_of = [&](const std::pair<int, int>& r) {
    long long c = 0;
    for (int b = r.first; b < r.second; ++b) c += P.buckets[b].chunks;
    return c;
  };
  auto by_size = [&](std::vector<std::pair<int, int>>& v) {
    std::stable_sort(v.begin(), v.end(), [&](const auto& x, const auto& y) {
      return chunks_of(x) < chunks_of(y);
    });
  };
  // buckets whose symmetric products cannot occupy every CTA pair (fewer tiles
  // than pairs) joined with their neighbour of the same form and orientation
  {
    auto small = [&](int b) {
      return (long long)P.buckets[b].mats.size() * (long long)P.buckets[b].sym.size() < clusters;
    };
    auto same = [&](int x, int y) {
      return P.buckets[x].tall == P.buckets[y].tall && P.buckets[x].gram == P.buckets[y].gram;
    };
    std::vector<std::pair<int, int>> merged;
    for (int b = 0; b < nb; ++b) {
      // a small bucket joins the position before it when that one is of the
      // same kind (and only one bucket long, or small itself), else starts one
      if (!merged.empty() && same(merged.back().first, b) && merged.back().second == b &&
          (small(b) || (merged.back().second - merged.back().first == 1 &&
                        small(merged.back().first))))
        merged.back().second = b + 1;
      else
        merged.push_back({b, b + 1});
    }
    if (int(merged.size()) < nb && merged.size() >= 2) {
      by_size(merged);
      cands.push_back(merged);
    }
  }
  std::vector<std::pair<int, int>> runs;
  for (int b = 0; b < nb;) {
    int e = b + 1;
    while (e < nb && P.buckets[e].tall == P.buckets[b].tall && P.buckets[e].gram == P.buckets[b].gram)
      ++e;
    runs.push_back({b, e});
    b = e;
  }
  if (runs.size() >= 2 && int(runs.size()) < nb) {
    by_size(runs);
    cands.push_back(runs);
  }
  StepSchedule best;
  bool have = false;
  for (const auto& c : cands) {
    StepSchedule S = plan_step(P, R, c, clusters);
    if (!have || S.products + S.exposed < best.products + best.exposed) {
      best = std::move(S);
      have = true;
    }
  }
  return best;
}

// Events used to order the two streams of an overlapped step; released when
// the call returns (the CUDA driver keeps a pending event alive until it fires).
struct EventSet {
  std::vector<cudaEvent_t> e;
  bool create(int count) {
    e.reserve(size_t(count));
    for (int i = 0; i < count; ++i) {
      cudaEvent_t x = nullptr;
      if (cudaEventCreateWithFlags(&x, cudaEventDisableTiming) != cudaSuccess) return false;
      e.push_back(x);
    }
    return true;
  }
  ~EventSet() {
    for (cudaEvent_t x : e) cudaEventDestroy(x);
  }
};

int run(const Request& R) {
  if (R.n < 0 || (R.n > 0 && R.shp == nullptr)) return DMUON_ERR_INVALID_ARG;
  // a pending, non-sticky error of earlier work on this thread is not ours:
  // clear it, so that the launch checks below report only this call's failures
  (void)cudaGetLastError();
  Plan P;
  int st = build_plan(R.n, R.shp, R.variant, R.ns_steps, P);
  if (st != DMUON_OK) return st;
  st = check_request(R, P);
  if (st != DMUON_OK) return st;
  if (R.n == 0) return DMUON_OK;
  DevInfo D;
  st = device_info(&D);
  if (st != DMUON_OK) return st;
  if (tensor_map_encoder() == nullptr) return DMUON_ERR_CUDA;
  st = upload_tables(R, P);
  if (st != DMUON_OK) return st;

  unsigned char* ws = static_cast<unsigned char*>(R.ws);
  const EwMat* ew = reinterpret_cast<const EwMat*>(ws + P.off_ew);
  float* partials = reinterpret_cast<float*>(ws + P.off_partials);
  float* inv = reinterpret_cast<float*>(ws + P.off_inv);
  __nv_bfloat16* packed = static_cast<__nv_bfloat16*>(R.packed);
  cudaStream_t s = R.stream;
  const bool gbf16 = R.grad_dt == DMUON_BF16, wbf16 = R.weight_dt == DMUON_BF16;
  const int nb = int(P.buckets.size());

  // the whole table, and the part of it that belongs to buckets [b0, b1)
  EwRange all{ew, R.n, 0, 0, P.total_chunks};
  auto range_of = [&](int b0, int b1) {
    EwRange r{ew + P.buckets[b0].first, 0, P.buckets[b0].first, P.buckets[b0].chunk_lo, 0};
    for (int b = b0; b < b1; ++b) {
      r.n += int(P.buckets[b].mats.size());
      r.chunks += P.buckets[b].chunks;
    }
    return r;
  };

  // A whole standard step over two or more buckets overlaps its memory-bound
  // work with the products (see choose_step_schedule and plan_step).
  const bool overlap = R.do_pack && R.do_ns && R.do_update && R.ns_steps > 0 && nb >= 2 &&
                       D.aux != nullptr;
  if (overlap) {
    const StepSchedule S = choose_step_schedule(P, R, D.max_clusters);
    const int g = int(S.pos.size());
    cudaStream_t x = aux_stream_for(D, s);
    size_t n_slots = 0;
    for (const auto& v : S.slot)
      for (const auto& w : v) n_slots += w.empty() ? 0 : 1;
    EventSet ev;  // [0, g): position k's pack done on aux; g: aux done; then one per used slot
    if (!ev.create(g + 1 + int(n_slots))) return DMUON_ERR_CUDA;
    size_t next_ev = size_t(g) + 1;
    auto bucket_range = [&](int b) { return range_of(b, b + 1); };
    std::vector<int> pos_of(static_cast<size_t>(nb), 0);
    for (int k = 0; k < g; ++k)
      for (int b = S.pos[size_t(k)].first; b < S.pos[size_t(k)].second; ++b) pos_of[size_t(b)] = k;
    // one piece of memory-bound work on stream `st`; pack work of a position
    // that runs on the aux stream records the position's event after it, so
    // that the caller's stream can wait for all of it before the position's
    // products (the last record before that wait is the one that counts)
    std::vector<char> aux_pack(static_cast<size_t>(g), 0);
    auto run_piece = [&](const Piece& pc, cudaStream_t st) {
      EwRange r = bucket_range(pc.bucket);
      bool ok = true;
      switch (pc.kind) {
        case kPiecePack:
          r.chunk_base += pc.lo;
          r.chunks = pc.hi - pc.lo;
          ok = launch_momentum_pack(r, gbf16, R.beta, packed, partials, st) == cudaSuccess;
          break;
        case kPieceFinalize:
          ok = launch_norm_finalize(r, partials, R.eps, inv, st) == cudaSuccess;
          break;
        case kPieceRelayout:
          r.chunk_base += pc.lo;
          r.chunks = pc.hi - pc.lo;
          ok = launch_relayout(r, packed, inv, st) == cudaSuccess;
          break;
        default:
          r.chunk_base += pc.lo;
          r.chunks = pc.hi - pc.lo;
          return launch_update(r, wbf16, R.lr, packed, st) == cudaSuccess;
      }
      if (ok && st == x) {
        const int k = pos_of[size_t(pc.bucket)];
        aux_pack[size_t(k)] = 1;
        ok = cudaEventRecord(ev.e[size_t(k)], x) == cudaSuccess;
      }
      return ok;
    };
    for (int k = 0; k < g; ++k) {
      if (aux_pack[size_t(k)] && cudaStreamWaitEvent(s, ev.e[size_t(k)], 0) != cudaSuccess)
        return DMUON_ERR_CUDA;
      for (const Piece& pc : S.pre[size_t(k)])
        if (!run_piece(pc, s)) return DMUON_ERR_CUDA;
      auto before = [&](int i) {
        const auto& pieces = S.slot[size_t(k)][size_t(i)];
        if (pieces.empty()) return true;
        // the pieces start together with this product launch
        cudaEvent_t e = ev.e[next_ev++];
        if (cudaEventRecord(e, s) != cudaSuccess || cudaStreamWaitEvent(x, e, 0) != cudaSuccess)
          return false;
        for (const Piece& pc : pieces)
          if (!run_piece(pc, x)) return false;
        return true;
      };
      const GemmLauncher L(P, R, D.max_clusters, ws, S.pos[size_t(k)].first,
                           S.pos[size_t(k)].second, s);
      if (!(P.buckets[S.pos[size_t(k)].first].gram ? ns_gram(L, R, before)
                                                   : ns_standard(L, R, P, ws, before)))
        return DMUON_ERR_CUDA;
    }
    for (const Piece& t : S.tail_update) {
      EwRange r = bucket_range(t.bucket);
      r.chunk_base += t.lo;
      r.chunks = t.hi - t.lo;
      if (launch_update(r, wbf16, R.lr, packed, s) != cudaSuccess) return DMUON_ERR_CUDA;
    }
    // join: only if anything ran on the aux stream (under stream capture, an
    // aux stream that never forked from `s` is not part of the capture)
    if (n_slots > 0 && (cudaEventRecord(ev.e[size_t(g)], x) != cudaSuccess ||
                        cudaStreamWaitEvent(s, ev.e[size_t(g)], 0) != cudaSuccess))
      return DMUON_ERR_CUDA;
    return DMUON_OK;
  }

  if (R.do_pack) {
    if (launch_momentum_pack(all, gbf16, R.beta, packed, partials, s) != cudaSuccess)
      return DMUON_ERR_CUDA;
  }
  if (R.do_ns) {
    if (!R.do_pack && !R.pack_norms) {
      if (launch_norm_partials(all, packed, partials, s) != cudaSuccess) return DMUON_ERR_CUDA;
    }
    if (launch_norm_finalize(all, partials, R.eps, inv, s) != cudaSuccess) return DMUON_ERR_CUDA;
    if (R.ns_steps == 0) {
      if (launch_scale_inplace(all, packed, inv, s) != cudaSuccess) return DMUON_ERR_CUDA;
    } else {
      if (launch_relayout(all, packed, inv, s) != cudaSuccess) return DMUON_ERR_CUDA;
      if (P.n_std > 0 &&
          !ns_standard(GemmLauncher(P, R, D.max_clusters, ws, 0, P.n_std, s), R, P, ws))
        return DMUON_ERR_CUDA;
      if (P.n_std < nb && !ns_gram(GemmLauncher(P, R, D.max_clusters, ws, P.n_std, nb, s), R))
        return DMUON_ERR_CUDA;
    }
  }
  if (R.do_update) {
    if (launch_update(all, wbf16, R.lr, packed, s) != cudaSuccess) return DMUON_ERR_CUDA;
  }
  return DMUON_OK;
}

}  // namespace
}  // namespace dm

namespace dm {
namespace {
thread_local long long t_launches = 0;
}  // namespace
void note_launch(int kernels) { t_launches += kernels; }
}  // namespace dm

// Built-in scratch of dmuon_ns_batched_noalloc.  Host code may not use the
// array's name as an address: the device address comes from
// cudaGetSymbolAddress, once per device.
static __device__ __align__(256) unsigned char g_noalloc_scratch[DMUON_NOALLOC_SCRATCH_BYTES];

namespace dm {
namespace {
void* g_noalloc_ptr[kMaxDevices] = {};

// Device address of the scratch array on the current device (null on error).
void* noalloc_scratch() {
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess || d < 0 || d >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lk(g_mu);
  if (g_noalloc_ptr[d] == nullptr) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
    g_noalloc_ptr[d] = p;
  }
  return g_noalloc_ptr[d];
}
}  // namespace
}  // namespace dm

using namespace dm;

extern "C" {

int dmuon_ns_batched_noalloc(int n, const dmuon_shape* shp, void* packed_bf16,
                             const int64_t* offset, int ns_steps, int ns_variant,
                             const float* abc, float eps, cudaStream_t stream) {
  Request R;
  R.n = n; R.shp = shp; R.packed = packed_bf16; R.offset = offset; R.ns_steps = ns_steps;
  R.variant = ns_variant;
  if (abc != nullptr) { R.abc[0] = abc[0]; R.abc[1] = abc[1]; R.abc[2] = abc[2]; }
  R.eps = eps; R.pack_norms = false; R.stream = stream; R.do_ns = true;
  // host-side checks first: nothing is enqueued for a rejected call
  if (n < 0 || (n > 0 && shp == nullptr)) return DMUON_ERR_INVALID_ARG;
  Plan P;
  int st = build_plan(n, shp, ns_variant, ns_steps, P);
  if (st != DMUON_OK) return st;
  if (P.total > size_t(DMUON_NOALLOC_SCRATCH_BYTES)) return DMUON_ERR_WORKSPACE;
  if (n == 0) return DMUON_OK;
  DevInfo D;
  st = device_info(&D);
  if (st != DMUON_OK) return st;
  void* scratch = noalloc_scratch();
  if (scratch == nullptr) return DMUON_ERR_CUDA;
  R.ws = scratch;
  R.ws_bytes = DMUON_NOALLOC_SCRATCH_BYTES;
  st = check_request(R, P);
  if (st != DMUON_OK) return st;
  // the device error word must start at zero; everything else in the scratch
  // is written before it is read
  if (cudaMemsetAsync(scratch, 0, sizeof(int), stream) != cudaSuccess) return DMUON_ERR_CUDA;
  return run(R);
}

int dmuon_noalloc_status(cudaStream_t stream) {
  void* scratch = noalloc_scratch();
  if (scratch == nullptr) return DMUON_ERR_CUDA;
  return dmuon_stream_status(stream, scratch);
}

int dmuon_plan(int n, const dmuon_shape* shp, int n_owners, int* owner_of, int64_t* offset,
               int64_t* owner_elems) {
  if (n < 0 || n_owners <= 0) return DMUON_ERR_INVALID_ARG;
  if (n > 0 && (shp == nullptr || owner_of == nullptr || offset == nullptr))
    return DMUON_ERR_INVALID_ARG;
  if (owner_elems == nullptr) return DMUON_ERR_INVALID_ARG;
  std::vector<int64_t> size(n);
  for (int i = 0; i < n; ++i) {
    if (!shape_ok(shp[i])) return DMUON_ERR_INVALID_ARG;
    size[i] = shp[i].rows * shp[i].cols;
  }
  // greedy LPT: descending size (ties: lower index), least-loaded owner (ties: lower owner)
  std::vector<int> order(n);
  for (int i = 0; i < n; ++i) order[i] = i;
  std::stable_sort(order.begin(), order.end(),
                   [&](int a, int b) { return size[a] > size[b]; });
  std::vector<int64_t> load(n_owners, 0);
  for (int i : order) {
    int best = 0;
    if (n_owners > 1)
      for (int o = 1; o < n_owners; ++o)
        if (load[o] < load[best]) best = o;
    owner_of[i] = n_owners > 1 ? best : 0;
    load[owner_of[i]] += size[i];
  }
  int64_t base = 0;
  for (int o = 0; o < n_owners; ++o) {
    int64_t cur = 0;
    for (int i = 0; i < n; ++i) {
      if (owner_of[i] != o) continue;
      offset[i] = base + cur;
      cur = int64_t(align_up(size_t(cur + size[i]), DMUON_PACK_ALIGN_ELEMS));
    }
    owner_elems[o] = cur;
    base += cur;
  }
  return DMUON_OK;
}

size_t dmuon_workspace_bytes(int n, const dmuon_shape* shp, int ns_variant) {
  // Which matrices run the Gram form depends on ns_steps: size for every step
  // count the rule distinguishes (1 and kGramMaxSteps + 1 stand for all others).
  size_t most = 0;
  const int last = ns_variant == DMUON_NS_GRAM ? kGramMaxSteps + 1 : 1;
  for (int k = 1; k <= last; ++k) {
    Plan P;
    if (build_plan(n, shp, ns_variant, k, P) != DMUON_OK) return 0;
    most = std::max(most, P.total);
  }
  return most;
}

int dmuon_ns_variant_for(int64_t rows, int64_t cols, int ns_steps, int ns_variant) {
  const dmuon_shape s{rows, cols};
  if (!shape_ok(s) || ns_steps < 0 || ns_steps > kMaxNsSteps || !variant_ok(ns_variant))
    return DMUON_ERR_INVALID_ARG;
  if (rows == 0 || cols == 0) return DMUON_NS_STANDARD;
  const int m = int(std::min(rows, cols)), nn = int(std::max(rows, cols));
  return uses_gram(ns_variant, m, nn, ns_steps) ? DMUON_NS_GRAM : DMUON_NS_STANDARD;
}

int dmuon_pack(int n, const dmuon_shape* shp, const void* const* grad, int grad_dt,
               float* const* momentum, float beta, void* packed_bf16, const int64_t* offset,
               void* workspace, size_t ws_bytes, cudaStream_t stream) {
  Request R;
  R.n = n; R.shp = shp; R.grad = grad; R.grad_dt = grad_dt; R.momentum = momentum;
  R.beta = beta; R.packed = packed_bf16; R.offset = offset; R.ws = workspace;
  R.ws_bytes = ws_bytes; R.stream = stream; R.do_pack = true;
  return run(R);
}

int dmuon_ns_batched(int n, const dmuon_shape* shp, void* packed_bf16, const int64_t* offset,
                     int ns_steps, int ns_variant, const float* abc, float eps,
                     int use_pack_norms, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  Request R;
  R.n = n; R.shp = shp; R.packed = packed_bf16; R.offset = offset; R.ns_steps = ns_steps;
  R.variant = ns_variant;
  if (abc != nullptr) { R.abc[0] = abc[0]; R.abc[1] = abc[1]; R.abc[2] = abc[2]; }
  R.eps = eps; R.pack_norms = use_pack_norms != 0; R.ws = workspace; R.ws_bytes = ws_bytes;
  R.stream = stream; R.do_ns = true;
  return run(R);
}

int dmuon_unpack_update(int n, const dmuon_shape* shp, void* const* weight, int weight_dt,
                        float lr, const void* packed_bf16, const int64_t* offset, void* workspace,
                        size_t ws_bytes, cudaStream_t stream) {
  Request R;
  R.n = n; R.shp = shp; R.weight = weight; R.weight_dt = weight_dt; R.lr = lr;
  R.packed = const_cast<void*>(packed_bf16); R.offset = offset; R.ws = workspace;
  R.ws_bytes = ws_bytes; R.stream = stream; R.do_update = true;
  return run(R);
}

int dmuon_muon_step(int n, const dmuon_shape* shp, const void* const* grad, int grad_dt,
                    float* const* momentum, void* const* weight, int weight_dt, float lr,
                    float beta, int ns_steps, int ns_variant, void* packed_bf16,
                    const int64_t* offset, void* workspace, size_t ws_bytes,
                    cudaStream_t stream) {
  Request R;
  R.n = n; R.shp = shp; R.grad = grad; R.grad_dt = grad_dt; R.momentum = momentum;
  R.weight = weight; R.weight_dt = weight_dt; R.lr = lr; R.beta = beta; R.ns_steps = ns_steps;
  R.variant = ns_variant; R.packed = packed_bf16; R.offset = offset; R.ws = workspace;
  R.ws_bytes = ws_bytes; R.stream = stream;
  R.do_pack = R.do_ns = R.do_update = true;
  R.pack_norms = true;
  return run(R);
}

size_t dmuon_adamw_workspace_bytes(int n) {
  if (n < 0) return 0;
  return align_up(kHdrBytes + size_t(n) * sizeof(AdamTensor), 256);
}

int dmuon_adamw(int n, const int64_t* numel, void* const* param, int param_dt,
                const void* const* grad, int grad_dt, float* const* exp_avg,
                float* const* exp_avg_sq, double lr, double beta1, double beta2, double eps,
                double weight_decay, int step, void* workspace, size_t ws_bytes,
                cudaStream_t stream) {
  if (n < 0) return DMUON_ERR_INVALID_ARG;
  if (n == 0) return DMUON_OK;
  if (numel == nullptr || param == nullptr || grad == nullptr || exp_avg == nullptr ||
      exp_avg_sq == nullptr || workspace == nullptr)
    return DMUON_ERR_INVALID_ARG;
  if ((param_dt != DMUON_F32 && param_dt != DMUON_BF16) ||
      (grad_dt != DMUON_F32 && grad_dt != DMUON_BF16))
    return DMUON_ERR_INVALID_ARG;
  if (step < 1 || !std::isfinite(lr) || !std::isfinite(eps) || !std::isfinite(weight_decay) ||
      !(beta1 >= 0.0 && beta1 < 1.0) || !(beta2 >= 0.0 && beta2 < 1.0) || !(eps >= 0.0))
    return DMUON_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return DMUON_ERR_ALIGNMENT;
  if (ws_bytes < dmuon_adamw_workspace_bytes(n)) return DMUON_ERR_WORKSPACE;
  std::vector<AdamTensor> ts(static_cast<size_t>(n));
  long long chunks = 0;
  for (int i = 0; i < n; ++i) {
    if (numel[i] < 0) return DMUON_ERR_INVALID_ARG;
    AdamTensor& T = ts[i];
    T.numel = numel[i];
    T.chunk_begin = chunks;
    chunks += ceil_div(numel[i], kChunk);
    if (numel[i] == 0) continue;
    if (param[i] == nullptr || grad[i] == nullptr || exp_avg[i] == nullptr ||
        exp_avg_sq[i] == nullptr)
      return DMUON_ERR_INVALID_ARG;
    T.p = param[i];
    T.g = grad[i];
    T.m = exp_avg[i];
    T.v = exp_avg_sq[i];
    T.vec = (aligned(T.p, 16) && aligned(T.g, 16) && aligned(T.m, 16) && aligned(T.v, 16)) ? 1 : 0;
  }
  if (chunks == 0) return DMUON_OK;
  DevInfo D;
  const int st = device_info(&D);
  if (st != DMUON_OK) return st;
  unsigned char* ws = static_cast<unsigned char*>(workspace);
  const size_t bytes = align_up(size_t(n) * sizeof(AdamTensor), 16);
  std::vector<unsigned char> blob(bytes, 0);
  std::memcpy(blob.data(), ts.data(), size_t(n) * sizeof(AdamTensor));
  if (launch_upload(ws + kHdrBytes, blob.data(), bytes, stream) != cudaSuccess)
    return DMUON_ERR_CUDA;
  // per-step scalars in double on the host, each rounded to fp32 once
  const double bc1 = 1.0 - std::pow(beta1, double(step));
  const double bc2 = 1.0 - std::pow(beta2, double(step));
  AdamScalars k;
  k.b1 = float(beta1);
  k.b2 = float(beta2);
  k.omb1 = float(1.0 - beta1);
  k.omb2 = float(1.0 - beta2);
  k.step_size = float(lr / bc1);
  k.inv_bc2_sqrt = float(1.0 / std::sqrt(bc2));
  k.eps = float(eps);
  k.decay = float(1.0 - lr * weight_decay);
  if (launch_adamw(reinterpret_cast<const AdamTensor*>(ws + kHdrBytes), n, chunks,
                   param_dt == DMUON_BF16, grad_dt == DMUON_BF16, k, stream) != cudaSuccess)
    return DMUON_ERR_CUDA;
  return DMUON_OK;
}

int dmuon_stream_status(cudaStream_t stream, void* workspace) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return DMUON_ERR_CUDA;
  if (workspace == nullptr) return DMUON_OK;
  if (!aligned(workspace, 256)) return DMUON_ERR_ALIGNMENT;
  int err = 0;
  if (cudaMemcpyAsync(&err, workspace, sizeof(int), cudaMemcpyDeviceToHost, stream) !=
          cudaSuccess ||
      cudaStreamSynchronize(stream) != cudaSuccess)
    return DMUON_ERR_CUDA;
  if (err != 0) {
    if (cudaMemsetAsync(workspace, 0, sizeof(int), stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess)
      return DMUON_ERR_CUDA;
    return err;
  }
  return DMUON_OK;
}

int dmuon_debug_wait_timeout(void* workspace, size_t ws_bytes, int budget_us,
                             cudaStream_t stream) {
  if (workspace == nullptr) {
    // the error word of dmuon_ns_batched_noalloc's built-in scratch
    workspace = noalloc_scratch();
    if (workspace == nullptr) return DMUON_ERR_CUDA;
    ws_bytes = DMUON_NOALLOC_SCRATCH_BYTES;
  }
  if (ws_bytes < kHdrBytes) return DMUON_ERR_INVALID_ARG;
  if (!aligned(workspace, 256)) return DMUON_ERR_ALIGNMENT;
  if (budget_us < 1 || budget_us > 1000000) return DMUON_ERR_INVALID_ARG;
  DevInfo D;
  const int st = device_info(&D);
  if (st != DMUON_OK) return st;
  const long long cycles = (long long)budget_us * (long long)D.clock_khz / 1000;
  if (launch_wait_timeout(static_cast<int*>(workspace), cycles, stream) != cudaSuccess)
    return DMUON_ERR_CUDA;
  return DMUON_OK;
}

static_assert(sizeof(dmuon_trace_record) == sizeof(TraceRec), "trace record layout");

int dmuon_trace_begin(void* records, size_t bytes) {
  if (records == nullptr || bytes < sizeof(TraceRec)) return DMUON_ERR_INVALID_ARG;
  if (!aligned(records, 16)) return DMUON_ERR_ALIGNMENT;
  int d = 0;
  if (cudaGetDevice(&d) != cudaSuccess) return DMUON_ERR_CUDA;
  trace_begin(records, bytes / sizeof(TraceRec), d);
  return DMUON_OK;
}

long long dmuon_trace_end(void) { return trace_end(); }

const char* dmuon_status_string(int status) {
  switch (status) {
    case DMUON_OK: return "ok";
    case DMUON_ERR_INVALID_ARG: return "invalid argument";
    case DMUON_ERR_ALIGNMENT: return "misaligned pointer or offset";
    case DMUON_ERR_WORKSPACE: return "workspace too small";
    case DMUON_ERR_CUDA: return "CUDA error";
    case DMUON_ERR_TIMEOUT: return "bounded device wait timed out";
    case DMUON_ERR_UNSUPPORTED: return "unsupported device or shape";
    default: return "unknown status";
  }
}

int dmuon_version(void) { return 100; }

long long dmuon_launch_count(int reset) {
  const long long n = t_launches;
  if (reset) t_launches = 0;
  return n;
}

}  // extern "C"
