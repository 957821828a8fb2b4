// flce_api.cu -- the C ABI (include/flce.h): argument checks, workspace layout,
// tensor-map encoding and the launch sequence of the forward and backward passes.
//
// Forward  ("Cutting LLM Memory by 84%", "Definition and Forward Pass"; Liger-Kernel
//           PR #1291 "Summary", store-free forward):
//   1. tensor-core GEMM over (cluster row block, vocabulary chunk) units, walked panel by
//      panel so that concurrent clusters share X rows and W tiles in L2, with the
//      online-softmax epilogue -> partial (max, sum-exp, sum-z) per row and chunk, target
//      logit;
//   2. finalize: combine the partials -> lse, row losses, deterministic reduction.
// Backward ("Backward Pass" and "Path to Production" of the same post; PR #1291: dW
//           contracts over the tokens and is written once):
//   1. prep: number of valid rows, g (over the whole batch), per-row coefficients; with
//      a 16-bit dX, the valid rows' X and coefficients are gathered to the front of the
//      (row band's) dX buffer (ignored rows have a zero gradient, so the GEMMs below skip
//      them) and the GEMMs read the device's row count;
//   2. for every band of Vc vocabulary columns (Vc picked so that the dW launches fill
//      whole waves of resident clusters), and for every row band when row_band is set:
//        gradient GEMM : recompute the logits, G = dZ in bf16 (f16: scaled) into the band;
//        dW GEMM       : dW[:, band] = X^T G   (K = rows, each block written once; later
//                        row bands, or accumulate_grads, add into it);
//        dX GEMM       : dX_acc (+)= G W[:, band]^T (fp32, TMA element-wise add);
//   3. cast dX_acc to bf16 (or f16) -- back to the original rows, zeros for ignored ones,
//      after a compaction -- unless the caller asked for the fp32 dX.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <initializer_list>
#include <mutex>

#include <cudaTypedefs.h>

#include "../../include/flce.h"
#include "flce_internal.h"

using namespace flce;

namespace {

// Compile-time tunables (defaults are the measured choices).
#ifndef FLCE_BAND_BYTES
// Byte budget of the 16-bit gradient band: 768 MiB keeps the backward's workspace (band +
// fp32 dX accumulator) under an eighth of the bf16 logits at N = 65536, V = 128256.
#define FLCE_BAND_BYTES (int64_t(3) << 28)
#endif
#ifndef FLCE_BAND_W_L2_BYTES
#define FLCE_BAND_W_L2_BYTES int64_t(0)  // if > 0: also cap the band so its W slice (2*D*Vc) fits this
#endif
#ifndef FLCE_BAND_PICK
#define FLCE_BAND_PICK 1  // 1: pick the band width for even dW waves; 0: the workspace's capacity
#endif
#ifndef FLCE_DW_TRANSPOSE_ODD
#define FLCE_DW_TRANSPOSE_ODD 1  // 1: G^T X with a transposed store when D's row tiles are odd
#endif
#ifndef FLCE_L2_PROMOTION
#define FLCE_L2_PROMOTION 3  // tensor-map L2 promotion: 0 none, 1 64 B, 2 128 B, 3 256 B
#endif
#ifndef FLCE_COMPACT_ROWS
#define FLCE_COMPACT_ROWS 1  // 1: the GEMMs skip ignored rows (valid-row compaction; the forward with room for it)
#endif

constexpr size_t kHeaderBytes = 256;
constexpr int64_t kGradBandBudget = FLCE_BAND_BYTES;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }
int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct FwdLayout {
  size_t part_m, part_d, part_s, part_idx, tgt, pred, block_sum, block_wsum, block_cnt, block_correct, total;
  int S_alloc, blocks;
};

// Header words of every workspace: [0] device error word, [8] number of valid rows
// (backward compaction), [16] B = g eps / V (backward), [24] sum of the class weights,
// [28] g (backward), [192] the forward GEMM's unit ticket counter. Bytes 32..159 hold
// the pipeline-wait counters of the diagnostic build.
constexpr size_t kHdrErr = 0, kHdrNValid = 8, kHdrB = 16, kHdrWtot = 24, kHdrG = 28, kHdrTicket = 192;

FwdLayout fwd_layout(int64_t N, int64_t V) {
  FwdLayout L{};
  const int64_t v_tiles = cdiv(V, kBN);
  L.S_alloc = int(v_tiles < kMaxSplits ? v_tiles : kMaxSplits);
  L.blocks = int(cdiv(N, kFinalizeThreads));
  size_t o = kHeaderBytes;
  const size_t part = align256(size_t(L.S_alloc) * size_t(N) * sizeof(float));
  L.part_m = o; o += part;
  L.part_d = o; o += part;
  L.part_s = o; o += part;
  L.part_idx = o; o += part;
  L.tgt = o; o += align256(size_t(N) * sizeof(float));
  L.pred = o; o += align256(size_t(N) * sizeof(int));
  L.block_sum = o; o += align256(size_t(L.blocks) * sizeof(double));
  L.block_wsum = o; o += align256(size_t(L.blocks) * sizeof(double));
  L.block_cnt = o; o += align256(size_t(L.blocks) * sizeof(int));
  L.block_correct = o; o += align256(size_t(L.blocks) * sizeof(int));
  L.total = o;
  return L;
}

// With room for it (flce_workspace_size(..., 3) bytes: any backward workspace has it), the
// forward runs its GEMM on the valid rows only: the row list, each row's slot, and the
// valid rows of X gathered (then zero rows up to the padding) follow the forward layout.
struct FwdCompactLayout {
  size_t rows, slot, xc, total;
};

FwdCompactLayout fwd_compact_layout(int64_t N, int64_t D, int64_t V) {
  FwdCompactLayout C{};
  size_t o = fwd_layout(N, V).total;
  C.rows = o; o += align256(size_t(N) * sizeof(int));
  C.slot = o; o += align256(size_t(N) * sizeof(int));
  C.xc = o; o += align256(size_t(N) * size_t(D) * 2);
  C.total = o;
  return C;
}

constexpr int kColsumChunks = 64;

struct BwdLayout {
  size_t coef, coef_c, rows, slot, band, dx_acc, colsum, total;
  int64_t Vc;
};

// Width of the gradient band: a multiple of one cluster's vocabulary tiles (2 pairs x 256
// rows when dW is [V, D], so no tile of a band reaches into the next), as many as fit in
// the byte budget, at most kMaxBandCols (wider bands measured no faster and cost memory),
// and never more than half the vocabulary (rounded up to that unit), so that no buffer
// holds N x V values once V exceeds one unit.
constexpr int64_t kMaxBandCols = 16384;

int64_t band_width(int64_t N, int64_t D, int64_t V) {
  const int64_t unit = int64_t(gemm_tile_rows()) * gemm_pairs_per_cluster();
  int64_t vc = (kGradBandBudget / (2 * N)) / unit * unit;
  if (vc > kMaxBandCols) vc = kMaxBandCols;
  if (FLCE_BAND_W_L2_BYTES > 0) {
    const int64_t l2 = (FLCE_BAND_W_L2_BYTES / (2 * D)) / unit * unit;
    if (l2 < vc) vc = l2;
  }
  if (vc < unit) vc = unit;
  const int64_t half = cdiv(cdiv(V, 2), unit) * unit;
  if (vc > half) vc = half;
  return vc;
}

// The dW GEMM computes G^T X (tile rows = vocabulary, the pairs of a cluster on
// neighbouring vocabulary tiles) for a [V, D] dW, and also for a [D, V] dW when D's row
// tiles do not split evenly among a cluster's pairs (the extra pair would compute zeros);
// its epilogue then stores the tiles transposed. Otherwise it computes X^T G.
bool dw_vocab_rows(int64_t D, bool w_vd) {
  return w_vd || (FLCE_DW_TRANSPOSE_ODD && cdiv(D, gemm_tile_rows()) % gemm_pairs_per_cluster() != 0);
}

// Launch units (clusters' worth of tiles) of the dW GEMM over a band of vc columns.
int64_t dw_units(int64_t vc, int64_t D, bool vocab_rows) {
  const int64_t mc = gemm_pairs_per_cluster();
  if (vocab_rows) return cdiv(cdiv(vc, gemm_tile_rows()), mc) * cdiv(D, kBN);
  return cdiv(cdiv(D, gemm_tile_rows()), mc) * cdiv(vc, kBN);
}

// The band width the backward uses for `rows` rows on a device with `clusters` resident
// clusters: among the multiples of 512 in [cap/2, cap], the one with the least estimated
// dW time. The dW GEMM has few, long tiles (K = rows), so it runs in whole waves of
// `clusters` units: a band of 32 vocabulary tiles on 36 clusters (8 units each) takes 8
// waves for 7.1 waves of work. The estimate counts waves over all bands plus, per band,
// ~20 us of launch ramp and tail, i.e. 4000/rows of a wave (a dW unit moves through K at
// ~5 ns per row). The gradient and dX GEMMs have thousands of short tiles and do not
// care. Ties keep the wider band. The workspace is sized for `cap`.
int64_t pick_band_width(int64_t cap, int64_t rows, int64_t D, int64_t V, bool w_vd, int clusters) {
  const int64_t unit = int64_t(gemm_tile_rows()) * gemm_pairs_per_cluster();
  if (!FLCE_BAND_PICK || clusters <= 0 || rows <= 0) return cap;
  const double band_cost = 4000.0 / double(rows);
  int64_t best = cap;
  double best_cost = 0.0;
  for (int64_t vc = cap; vc >= unit && 2 * vc >= cap; vc -= unit) {
    int64_t waves = 0, bands = 0;
    for (int64_t v0 = 0; v0 < V; v0 += vc, ++bands)
      waves += cdiv(dw_units(V - v0 < vc ? V - v0 : vc, D, dw_vocab_rows(D, w_vd)), clusters);
    const double cost = double(waves) + band_cost * double(bands);
    if (vc == cap || cost < best_cost - 1e-9) {
      best_cost = cost;
      best = vc;
    }
  }
  return best;
}

BwdLayout bwd_layout(int64_t N, int64_t D, int64_t V) {
  BwdLayout L{};
  L.Vc = band_width(N, D, V);
  size_t o = kHeaderBytes;
  L.coef = o; o += align256(size_t(N) * 16);
  L.coef_c = o; o += align256(size_t(N) * 16);
  L.rows = o; o += align256(size_t(N) * sizeof(int));
  L.slot = o; o += align256(size_t(N) * sizeof(int));
  L.band = o; o += align256(size_t(N) * size_t(L.Vc) * 2);
  L.dx_acc = o; o += align256(size_t(N) * size_t(D) * sizeof(float));
  L.colsum = o; o += align256(size_t(kColsumChunks) * size_t(L.Vc) * sizeof(float));
  L.total = o;
  return L;
}

bool sizes_ok(int64_t N, int64_t D, int64_t V) { return N >= 1 && D >= 1 && V >= 1; }

bool sizes_in_range(int64_t N, int64_t D, int64_t V) {
  const int64_t lim = int64_t(1) << 30;
  return N < lim && D < lim && V < lim;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// --- the detail behind FLCE_ERR_CUDA (per calling thread) ---------------------------
thread_local char g_detail[192];

void note_error(const char* what, const char* why) {
  std::snprintf(g_detail, sizeof(g_detail), "%.120s: %.60s", what, why);
}

void note_cuda_error(const char* what, cudaError_t e) { note_error(what, cudaGetErrorName(e)); }

// --- device and driver entry points ---------------------------------------------
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
PFN_cuCtxGetCurrent_v4000 g_ctx_current = nullptr;
std::once_flag g_encode_once;

void* driver_entry(const char* name, int version) {
  void* fn = nullptr;
  cudaDriverEntryPointQueryResult q;
  if (cudaGetDriverEntryPointByVersion(name, &fn, version, cudaEnableDefault, &q) == cudaSuccess &&
      q == cudaDriverEntryPointSuccess)
    return fn;
  cudaGetLastError();
  return nullptr;
}

struct DevInfo {
  bool known;
  bool ok;
  int sms;
};
DevInfo g_dev[64];
std::mutex g_dev_mu;

flce_status current_device(int* sms, int* dev_out = nullptr) {
  int dev = -1;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0) {
    cudaGetLastError();
    return FLCE_ERR_UNSUPPORTED_DEVICE;
  }
  std::lock_guard<std::mutex> lock(g_dev_mu);
  if (dev >= 64) return FLCE_ERR_UNSUPPORTED_DEVICE;
  if (!g_dev[dev].known) {
    int major = 0, minor = 0, n = 0;
    bool ok = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) == cudaSuccess &&
              cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) == cudaSuccess &&
              cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) == cudaSuccess;
    if (!ok) cudaGetLastError();
    g_dev[dev].known = true;
    g_dev[dev].ok = ok && major == 10 && minor == 3;
    g_dev[dev].sms = n;
  }
  if (!g_dev[dev].ok) return FLCE_ERR_UNSUPPORTED_DEVICE;
  *sms = g_dev[dev].sms;
  if (dev_out) *dev_out = dev;
  std::call_once(g_encode_once, [] {
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(driver_entry("cuTensorMapEncodeTiled", 12000));
    g_ctx_current = reinterpret_cast<PFN_cuCtxGetCurrent_v4000>(driver_entry("cuCtxGetCurrent", 4000));
  });
  if (!g_encode || !g_ctx_current) {
    note_error("cudaGetDriverEntryPointByVersion", "cuTensorMapEncodeTiled or cuCtxGetCurrent not found");
    return FLCE_ERR_CUDA;
  }
  // A thread that has made no CUDA call yet (a framework's worker thread, say) has no
  // current context, and the tensor-map encoder, a driver call, needs one: bind the
  // device's primary context, as the runtime's own calls would. A context the caller
  // made current is left alone.
  CUcontext ctx = nullptr;
  if (g_ctx_current(&ctx) != CUDA_SUCCESS || ctx == nullptr) {
    const cudaError_t e = cudaSetDevice(dev);
    if (e != cudaSuccess) {
      note_cuda_error("cudaSetDevice", e);
      cudaGetLastError();
      return FLCE_ERR_CUDA;
    }
  }
  return FLCE_OK;
}

// Every buffer an entry point is given must be memory that device `dev` addresses as its
// own: device memory of that device, or managed memory. Host memory (pinned or pageable)
// and another device's memory are refused before anything is launched, since a kernel or
// a tensor-map copy on such an address would read over the host link or fault.
struct NamedPtr {
  const char* name;
  const void* p;
};

flce_status check_device_memory(int dev, std::initializer_list<NamedPtr> bufs) {
  for (const NamedPtr& b : bufs) {
    if (!b.p) continue;
    cudaPointerAttributes a{};
    const cudaError_t e = cudaPointerGetAttributes(&a, b.p);
    if (e != cudaSuccess) {
      cudaGetLastError();
      note_error(b.name, "memory kind unreadable (cudaPointerGetAttributes)");
      return FLCE_ERR_INVALID_ARG;
    }
    if (a.type == cudaMemoryTypeManaged || (a.type == cudaMemoryTypeDevice && a.device == dev)) continue;
    note_error(b.name, a.type == cudaMemoryTypeDevice ? "is memory of another device than the current one"
                                                      : "is host memory, not device memory");
    return FLCE_ERR_INVALID_ARG;
  }
  return FLCE_OK;
}

flce_status check_option_memory(int dev, const flce_options* o) {
  if (!o) return FLCE_OK;
  return check_device_memory(dev, {{"options.bias", o->bias},
                                   {"options.class_weight", o->class_weight},
                                   {"options.predicted", o->predicted},
                                   {"options.accuracy", o->accuracy},
                                   {"options.dbias", o->dbias},
                                   {"options.dX_f32", o->dX_f32}});
}

// 2-D row-major tensor [outer][inner] with row pitch `pitch_elems`, 128-byte swizzled boxes.
bool encode_2d(CUtensorMap* m, CUtensorMapDataType dt, int elem_bytes, const void* base, uint64_t inner,
               uint64_t outer, uint64_t pitch_elems, uint32_t box_inner, uint32_t box_outer,
               bool swizzle = true) {
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {pitch_elems * uint64_t(elem_bytes)};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return g_encode(m, dt, 2, const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                  swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
                  static_cast<CUtensorMapL2promotion>(FLCE_L2_PROMOTION),
                  CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS ||
         (note_error("cuTensorMapEncodeTiled", "the tensor map was refused"), false);
}

flce_status check_common(const void* X, const void* W, const int32_t* targets, int64_t N, int64_t D, int64_t V,
                         float eps, float s, int red, const void* ws) {
  if (!X || !W || !targets || !ws) return FLCE_ERR_INVALID_ARG;
  if (!sizes_ok(N, D, V)) return FLCE_ERR_INVALID_ARG;
  if (!(eps >= 0.f && eps < 1.f)) return FLCE_ERR_INVALID_ARG;
  if (!(s >= 0.f) || std::isinf(s)) return FLCE_ERR_INVALID_ARG;
  if (red < 0 || red > 2) return FLCE_ERR_INVALID_ARG;
  if (!sizes_in_range(N, D, V)) return FLCE_ERR_TOO_LARGE;
  if (D % 8 != 0 || V % 8 != 0) return FLCE_ERR_ALIGNMENT;
  if (!aligned(X, 16) || !aligned(W, 16) || !aligned(ws, 16) || !aligned(targets, 4)) return FLCE_ERR_ALIGNMENT;
  return FLCE_OK;
}

// The forward's units: cluster row blocks x vocabulary chunks (at most kMaxSplits chunks,
// so at most that many partial statistics per row), walked panel by panel.
void pick_forward_schedule(int64_t n_tiles, int64_t v_tiles, int64_t D, FwdParams* p) {
  const int64_t block_rows = int64_t(gemm_pairs_per_cluster()) * kFwdRowBlock * gemm_tile_rows();
  const int64_t n_blocks = cdiv(n_tiles, int64_t(gemm_pairs_per_cluster()) * kFwdRowBlock);
  const int64_t chunk_tiles = cdiv(v_tiles, kMaxSplits);
  const int64_t n_chunks = cdiv(v_tiles, chunk_tiles);
  int64_t panel = FLCE_FWD_PANEL > 0 ? int64_t(FLCE_FWD_PANEL) : FLCE_FWD_PANEL_BYTES / (block_rows * D * 2);
  if (panel < 1) panel = 1;
  p->n_blocks = int(n_blocks);
  p->panel = int(n_blocks < panel ? n_blocks : panel);
  p->chunk_tiles = int(chunk_tiles);
  p->n_chunks = int(n_chunks);
  p->total_units = int(n_blocks * n_chunks);
}

#define FLCE_CUDA_CHECK(expr)                    \
  do {                                           \
    const cudaError_t flce_e_ = (expr);          \
    if (flce_e_ != cudaSuccess) {                \
      note_cuda_error(#expr, flce_e_);           \
      cudaGetLastError();                        \
      return FLCE_ERR_CUDA;                      \
    }                                            \
  } while (0)

}  // namespace

extern "C" {

int flce_version(void) { return 300; }

const char* flce_last_error_detail(void) { return g_detail; }

unsigned long long flce_kernel_launches(void) { return launches_so_far(); }

void flce_profile_gemms(int enable) { profile_enable(enable != 0); }

flce_status flce_profile_read(double* ms, unsigned long long* launches) {
  if (!ms || !launches) return FLCE_ERR_INVALID_ARG;
  FLCE_CUDA_CHECK(profile_read(ms, launches));
  return FLCE_OK;
}

flce_status flce_selftest_wait_timeout(void* workspace, size_t ws_bytes, struct CUstream_st* stream_) {
  if (!workspace) return FLCE_ERR_INVALID_ARG;
  if (!aligned(workspace, 16)) return FLCE_ERR_ALIGNMENT;
  if (ws_bytes < kHeaderBytes) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  int sms = 0, dev = -1;
  flce_status st = current_device(&sms, &dev);
  if (st != FLCE_OK) return st;
  if ((st = check_device_memory(dev, {{"workspace", workspace}})) != FLCE_OK) return st;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  FLCE_CUDA_CHECK(cudaMemsetAsync(workspace, 0, kHeaderBytes, stream));
  FLCE_CUDA_CHECK(launch_wait_selftest(reinterpret_cast<int*>(static_cast<uint8_t*>(workspace) + kHdrErr), stream));
  return FLCE_OK;
}

const char* flce_status_string(flce_status st) {
  switch (st) {
    case FLCE_OK: return "FLCE_OK";
    case FLCE_ERR_INVALID_ARG: return "FLCE_ERR_INVALID_ARG: null pointer, bad size, option or enum";
    case FLCE_ERR_ALIGNMENT: return "FLCE_ERR_ALIGNMENT: D and V must be multiples of 8 and pointers aligned";
    case FLCE_ERR_UNSUPPORTED_DEVICE: return "FLCE_ERR_UNSUPPORTED_DEVICE: needs a compute capability 10.3 GPU";
    case FLCE_ERR_WORKSPACE_TOO_SMALL: return "FLCE_ERR_WORKSPACE_TOO_SMALL";
    case FLCE_ERR_REDUCTION_NONE_GRAD: return "FLCE_ERR_REDUCTION_NONE_GRAD: reduction 'none' has no fused backward";
    case FLCE_ERR_CUDA: return "FLCE_ERR_CUDA: a CUDA runtime or driver call failed";
    case FLCE_ERR_BAD_TARGET: return "FLCE_ERR_BAD_TARGET: a target outside [0, V) that is not ignore_index";
    case FLCE_ERR_TIMEOUT: return "FLCE_ERR_TIMEOUT: a device pipeline wait exceeded its limit";
    case FLCE_ERR_TOO_LARGE: return "FLCE_ERR_TOO_LARGE: a size exceeds 2^30";
    case FLCE_ERR_F16_RANGE: return "FLCE_ERR_F16_RANGE: an f16 gradient coefficient exceeds the f16 range";
  }
  return "unknown flce_status";
}

size_t flce_workspace_size(int64_t N, int64_t D, int64_t V, int for_backward) {
  if (!sizes_ok(N, D, V) || !sizes_in_range(N, D, V)) return 0;
  const size_t f = fwd_layout(N, V).total, b = bwd_layout(N, D, V).total;
  if (for_backward == 0) return f;
  if (for_backward == 1) return b;
  if (for_backward == 3) return fwd_compact_layout(N, D, V).total;
  return f > b ? f : b;
}

}  // extern "C"

namespace {

struct Problem {
  const void* X;
  const void* W;
  const int32_t* targets;
  int64_t N, D, V;
  int32_t ignore_index;
  float eps, zscale;
  flce_reduction red;
  bool w_vd;  // W (and dW) stored [V, D] (nn.Linear's weight layout); else [D, V]
  bool f16;   // X and W (and dX) are f16; else bf16
  // tensor-map element type of X, W and the gradient band
  CUtensorMapDataType dt16() const {
    return f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  }
};

bool opt_w_vd(const flce_options* o) { return o && o->weight_layout == FLCE_WEIGHT_VD; }
bool opt_f16(const flce_options* o) { return o && o->input_dtype == FLCE_INPUT_F16; }

bool opt_ext_forward(const flce_options* o) {
  return o && (o->softcap > 0.f || o->bias || o->class_weight || o->predicted || o->accuracy);
}

bool opt_ext_grad(const flce_options* o) { return o && (o->softcap > 0.f || o->bias || o->class_weight); }

flce_status check_options(const flce_options* o, const Problem& pb, bool backward) {
  if (!o) return FLCE_OK;
  if (!(o->softcap >= 0.f) || std::isinf(o->softcap)) return FLCE_ERR_INVALID_ARG;
  if ((o->bias && !aligned(o->bias, 4)) || (o->class_weight && !aligned(o->class_weight, 4)) ||
      (o->predicted && !aligned(o->predicted, 4)) || (o->accuracy && !aligned(o->accuracy, 4)) ||
      (o->dbias && !aligned(o->dbias, 4)) || (o->dX_f32 && !aligned(o->dX_f32, 16)))
    return FLCE_ERR_ALIGNMENT;
  if (o->dbias && !o->bias) return FLCE_ERR_INVALID_ARG;
  if (o->row_band < 0) return FLCE_ERR_INVALID_ARG;
  if (o->weight_layout != FLCE_WEIGHT_DV && o->weight_layout != FLCE_WEIGHT_VD) return FLCE_ERR_INVALID_ARG;
  if (o->input_dtype != FLCE_INPUT_BF16 && o->input_dtype != FLCE_INPUT_F16) return FLCE_ERR_INVALID_ARG;
  if (o->accumulate_grads != 0 && o->accumulate_grads != 1) return FLCE_ERR_INVALID_ARG;
  const bool shard = o->v_total != 0 && o->v_total != pb.V;
  if (shard) {
    if (!backward) return FLCE_ERR_INVALID_ARG;  // forward shards go through flce_shard_stats
    if (o->v_total < pb.V || o->v_offset < 0 || o->v_offset + pb.V > o->v_total) return FLCE_ERR_INVALID_ARG;
    if (o->v_total >= (int64_t(1) << 30)) return FLCE_ERR_TOO_LARGE;
    if (o->softcap > 0.f || o->bias || o->class_weight || o->dbias) return FLCE_ERR_INVALID_ARG;
  } else if (o->v_offset != 0) {
    return FLCE_ERR_INVALID_ARG;
  }
  return FLCE_OK;
}

// Forward GEMM + finalize. mode FIN_LOSS (loss, lse, options) or FIN_SHARD_STATS.
flce_status run_forward(const Problem& pb, const flce_options* opt, int mode, int64_t v_offset, float* loss,
                        float* lse, float* stats, uint8_t* ws, size_t ws_bytes, bool clear_header, int sms,
                        cudaStream_t stream) {
  const FwdLayout L = fwd_layout(pb.N, pb.V);
  int* err = reinterpret_cast<int*>(ws + kHdrErr);
  float* wtot = reinterpret_cast<float*>(ws + kHdrWtot);
  const int64_t n_tiles = cdiv(pb.N, gemm_tile_rows()), v_tiles = cdiv(pb.V, kBN);
  const bool ext = mode == FIN_LOSS && opt_ext_forward(opt);
  // Valid rows only (the plain epilogue; an ignored row's loss is 0 and its lse is not
  // needed): the GEMM reads the gathered valid rows of X, with room in the workspace.
  const FwdCompactLayout C = fwd_compact_layout(pb.N, pb.D, pb.V);
  // (from 2048 rows: below that the two extra launches cost more than the rows they save)
  const bool compact = FLCE_COMPACT_ROWS && mode == FIN_LOSS && !ext && ws_bytes >= C.total && pb.N >= 2048;

  // B = W: MN-major 64 x 64 boxes of W [D, V], or K-major boxes of W [V, D]
  CUtensorMap tmX, tmW;
  const bool enc_w =
      pb.w_vd ? encode_2d(&tmW, pb.dt16(), 2, pb.W, uint64_t(pb.D), uint64_t(pb.V), uint64_t(pb.D), 64,
                          uint32_t(gemm_b_rows_per_cta()))
              : encode_2d(&tmW, pb.dt16(), 2, pb.W, uint64_t(pb.V), uint64_t(pb.D), uint64_t(pb.V), 64, 64);
  const void* Xa = compact ? static_cast<const void*>(ws + C.xc) : pb.X;
  const bool enc_x =
      encode_2d(&tmX, pb.dt16(), 2, Xa, uint64_t(pb.D), uint64_t(pb.N), uint64_t(pb.D), 64, kBM);
  if (!enc_w || !enc_x) return FLCE_ERR_CUDA;

  if (clear_header) FLCE_CUDA_CHECK(cudaMemsetAsync(ws, 0, kHeaderBytes, stream));
  const float* cw = opt ? opt->class_weight : nullptr;
  if (cw) FLCE_CUDA_CHECK(launch_sum(cw, int(pb.V), wtot, stream));
  const bool want_idx = ext && (opt->predicted || opt->accuracy);
  int* n_valid = reinterpret_cast<int*>(ws + kHdrNValid);
  int* rows = reinterpret_cast<int*>(ws + C.rows);
  int* slot = reinterpret_cast<int*>(ws + C.slot);
  if (compact) {
    const CompactParams cp{pb.targets, int(pb.N), pb.ignore_index, rows, slot, n_valid};
    FLCE_CUDA_CHECK(launch_compact_rows(cp, stream));
    const GatherParams gp{pb.X, ws + C.xc, nullptr, nullptr, rows, n_valid, int(pb.N), int(pb.D)};
    FLCE_CUDA_CHECK(launch_gather_rows(gp, sms, stream));
  }

  FwdParams p{};
  p.targets = pb.targets;
  p.N = int(pb.N);
  p.V = int(pb.V);
  p.n_tiles = int(n_tiles);
  p.v_tiles = int(v_tiles);
  pick_forward_schedule(n_tiles, v_tiles, pb.D, &p);
  p.ticket = reinterpret_cast<int*>(ws + kHdrTicket);  // zeroed with the header above
  p.dyn_rows = compact ? n_valid : nullptr;
  p.row_of = compact ? rows : nullptr;
  if (!clear_header) FLCE_CUDA_CHECK(cudaMemsetAsync(p.ticket, 0, sizeof(int), stream));
  p.num_kb = int(cdiv(pb.D, kBK));
  p.want_sum_z = (mode == FIN_SHARD_STATS) || pb.eps != 0.f;
  p.ignore_index = pb.ignore_index;
  p.y_offset = int(v_offset);
  p.part_m = reinterpret_cast<float*>(ws + L.part_m);
  p.part_d = reinterpret_cast<float*>(ws + L.part_d);
  p.part_s = reinterpret_cast<float*>(ws + L.part_s);
  p.tgt = reinterpret_cast<float*>(ws + L.tgt);
  p.err = err;
  if (ext) {
    p.bias = opt->bias;
    p.cw = cw;
    p.softcap = opt->softcap;
    p.part_idx = want_idx ? reinterpret_cast<int*>(ws + L.part_idx) : nullptr;
  }
  FLCE_CUDA_CHECK(launch_forward_gemm(tmX, tmW, p, ext, pb.w_vd, pb.f16, stream));

  FinalizeParams f{};
  f.mode = mode;
  f.part_m = p.part_m;
  f.part_d = p.part_d;
  f.part_s = p.part_s;
  f.tgt = p.tgt;
  f.part_idx = p.part_idx;
  f.targets = pb.targets;
  f.N = int(pb.N);
  f.V = int(pb.V);
  f.S = p.n_chunks;
  f.V_local = int(pb.V);
  f.v_offset = int(v_offset);
  f.ignore_index = pb.ignore_index;
  f.eps = pb.eps;
  f.zscale = pb.zscale;
  f.reduction = int(pb.red);
  f.cw = ext ? cw : nullptr;
  f.wtot = wtot;
  f.lse = lse;
  f.slot = compact ? slot : nullptr;
  f.loss = loss;
  f.stats_out = stats;
  // The argmax decision is made per row in the finalize; without a caller array it
  // lands in scratch (accuracy only).
  f.predicted = want_idx ? (opt->predicted ? opt->predicted : reinterpret_cast<int*>(ws + L.pred)) : nullptr;
  f.accuracy = want_idx ? opt->accuracy : nullptr;
  f.block_sum = reinterpret_cast<double*>(ws + L.block_sum);
  f.block_wsum = reinterpret_cast<double*>(ws + L.block_wsum);
  f.block_cnt = reinterpret_cast<int*>(ws + L.block_cnt);
  f.block_correct = reinterpret_cast<int*>(ws + L.block_correct);
  f.err = err;
  FLCE_CUDA_CHECK(launch_finalize(f, L.blocks, stream));
  return FLCE_OK;
}

bool overlaps(const void* a, size_t a_bytes, const void* b, size_t b_bytes) {
  if (!a || !b) return false;
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + b_bytes && y < x + a_bytes;
}

// The valid-row compaction keeps its copy of X's valid rows in the caller's 16-bit dX
// buffer, which the backward otherwise writes only at its end: that buffer must not
// overlap anything the backward reads.
bool dx_free_for_scratch(const Problem& pb, const flce_options* opt, const float* lse, const float* grad_out,
                         const void* dX) {
  const size_t n = size_t(pb.N), d = size_t(pb.D), v = size_t(pb.V);
  const size_t bytes = n * d * 2;
  return !overlaps(dX, bytes, pb.X, n * d * 2) && !overlaps(dX, bytes, pb.W, d * v * 2) &&
         !overlaps(dX, bytes, pb.targets, n * 4) && !overlaps(dX, bytes, lse, n * 4) &&
         !overlaps(dX, bytes, grad_out, 4) && !(opt && overlaps(dX, bytes, opt->bias, v * 4)) &&
         !(opt && overlaps(dX, bytes, opt->class_weight, v * 4));
}

// Rows handled per backward pass: all of them, or bands of opt->row_band.
int64_t backward_rows(const flce_options* opt, int64_t N) {
  return (opt && opt->row_band > 0 && opt->row_band < N) ? opt->row_band : N;
}

flce_status run_backward(const Problem& pb, const flce_options* opt, const float* lse, const float* grad_out,
                         void* dX, float* dW, uint8_t* ws, bool clear_header, int sms, cudaStream_t stream) {
  const int64_t Nb = backward_rows(opt, pb.N);
  const BwdLayout L = bwd_layout(Nb, pb.D, pb.V);
  int* err = reinterpret_cast<int*>(ws + kHdrErr);
  float* bval = reinterpret_cast<float*>(ws + kHdrB);
  float* wtot = reinterpret_cast<float*>(ws + kHdrWtot);
  float* gval = reinterpret_cast<float*>(ws + kHdrG);
  float4* coef = reinterpret_cast<float4*>(ws + L.coef);
  void* band = ws + L.band;
  float* dx_acc = reinterpret_cast<float*>(ws + L.dx_acc);
  const bool f32_out = opt && opt->dX_f32;
  const int64_t Vc = pick_band_width(L.Vc, Nb, pb.D, pb.V, pb.w_vd, walk_max_clusters());
  const bool shard = opt && opt->v_total != 0 && opt->v_total != pb.V;
  const int64_t V_total = shard ? opt->v_total : pb.V;
  const int64_t v_offset = shard ? opt->v_offset : 0;
  const float* cw = opt ? opt->class_weight : nullptr;
  const bool ext = opt_ext_grad(opt);
  const float* out_scale = pb.f16 ? gval : nullptr;  // dW, dX = g / kF16GradScale * (f16 band GEMM)
  const bool add_grads = opt && opt->accumulate_grads;  // dW (and dbias) += this call's gradient
  // Valid-row compaction: an ignored row's gradient is zero, so the GEMMs take only the
  // valid rows, gathered into the row band's part of the 16-bit dX buffer.
  const bool compact = FLCE_COMPACT_ROWS && !f32_out && dx_free_for_scratch(pb, opt, lse, grad_out, dX);
  int* n_valid_dev = reinterpret_cast<int*>(ws + kHdrNValid);
  int* rows = reinterpret_cast<int*>(ws + L.rows);
  int* slot = reinterpret_cast<int*>(ws + L.slot);
  float4* coef_c = reinterpret_cast<float4*>(ws + L.coef_c);

  // Maps that do not depend on the row band. tmWg: B of the gradient GEMM (N = vocabulary,
  // K = D); tmWx: B of the dX GEMM (N = D, K = vocabulary). Each is MN-major in one W layout
  // and K-major in the other; K-major boxes are 64 x (rows per CTA), MN-major ones 64 x 64.
  const uint64_t w_inner = pb.w_vd ? uint64_t(pb.D) : uint64_t(pb.V);
  const uint64_t w_outer = pb.w_vd ? uint64_t(pb.V) : uint64_t(pb.D);
  const uint32_t kmaj_rows = uint32_t(gemm_b_rows_per_cta());
  CUtensorMap tmWg, tmWx, tmDW, tmDWt;
  if (!encode_2d(&tmWg, pb.dt16(), 2, pb.W, w_inner, w_outer, w_inner, 64,
                 pb.w_vd ? kmaj_rows : 64) ||
      !encode_2d(&tmWx, pb.dt16(), 2, pb.W, w_inner, w_outer, w_inner, 64,
                 pb.w_vd ? 64 : kmaj_rows) ||
      !encode_2d(&tmDW, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dW, w_inner, w_outer, w_inner, 32, kBM) ||
      // [D, V] dW written from G^T X tiles: 32 rows of D x 128 vocabulary columns, unswizzled
      !encode_2d(&tmDWt, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dW, w_inner, w_outer, w_inner, kBM, 32, false))
    return FLCE_ERR_CUDA;

  if (clear_header) FLCE_CUDA_CHECK(cudaMemsetAsync(ws, 0, kHeaderBytes, stream));
  if (cw) FLCE_CUDA_CHECK(launch_sum(cw, int(pb.V), wtot, stream));
  PrepParams pp{};
  pp.targets = pb.targets;
  pp.lse = lse;
  pp.grad_out = grad_out;
  pp.N = int(pb.N);
  pp.V = int(V_total);
  pp.y_offset = int(v_offset);
  pp.ignore_index = pb.ignore_index;
  pp.eps = pb.eps;
  pp.zscale = pb.zscale;
  pp.reduction = int(pb.red);
  pp.cw = cw;
  pp.wtot = wtot;
  pp.coef = coef;
  pp.gval = gval;
  pp.bval = bval;
  pp.gscale = pb.f16 ? kF16GradScale : 0.f;  // the f16 band holds G / g, scaled
  pp.err = err;
  FLCE_CUDA_CHECK(launch_denominator(pp, stream));  // g over every row of the batch

  const int64_t mc = gemm_pairs_per_cluster();
  const int64_t d_tiles_m = cdiv(cdiv(pb.D, gemm_tile_rows()), mc);  // dW [D, V]: row-tile groups
  const int64_t d_tiles_n = cdiv(pb.D, kBN);                         // dX columns
  for (int64_t n0 = 0; n0 < pb.N; n0 += Nb) {
    const int64_t nb = (pb.N - n0 < Nb) ? pb.N - n0 : Nb;
    // the GEMMs' X: this row band of X, or its valid rows compacted into the band's dX rows
    const size_t band_off = size_t(n0) * size_t(pb.D) * 2;
    const void* Xrows = static_cast<const uint8_t*>(pb.X) + band_off;
    void* dXrows = compact ? static_cast<uint8_t*>(dX) + band_off : nullptr;
    const void* Xb = compact ? static_cast<const void*>(dXrows) : Xrows;
    float* dx_dst = f32_out ? opt->dX_f32 + size_t(n0) * size_t(pb.D) : dx_acc;
    CUtensorMap tmXk, tmXmn, tmG, tmGmn, tmDX;
    const bool enc =
        encode_2d(&tmXk, pb.dt16(), 2, Xb, uint64_t(pb.D), uint64_t(nb), uint64_t(pb.D), 64,
                  kBM) &&
        encode_2d(&tmXmn, pb.dt16(), 2, Xb, uint64_t(pb.D), uint64_t(nb), uint64_t(pb.D), 64,
                  64) &&
        encode_2d(&tmG, pb.dt16(), 2, band, uint64_t(Vc), uint64_t(nb), uint64_t(Vc), 64,
                  kBM) &&
        encode_2d(&tmGmn, pb.dt16(), 2, band, uint64_t(Vc), uint64_t(nb), uint64_t(Vc), 64,
                  64) &&
        encode_2d(&tmDX, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 4, dx_dst, uint64_t(pb.D), uint64_t(nb), uint64_t(pb.D),
                  32, kBM);
    if (!enc) return FLCE_ERR_CUDA;
    PrepParams pb_rows = pp;
    pb_rows.targets = pb.targets + n0;
    pb_rows.lse = lse + n0;
    FLCE_CUDA_CHECK(launch_coef(pb_rows, int(nb), stream));
    const float4* coef_rows = coef;
    const int* dyn = nullptr;
    if (compact) {
      const CompactParams cp{pb.targets + n0, int(nb), pb.ignore_index, rows, slot, n_valid_dev};
      FLCE_CUDA_CHECK(launch_compact_rows(cp, stream));
      const GatherParams gp{Xrows, dXrows, coef, coef_c, rows, n_valid_dev, int(nb), int(pb.D)};
      FLCE_CUDA_CHECK(launch_gather_rows(gp, sms, stream));
      coef_rows = coef_c;
      dyn = n_valid_dev;
    }

    const int64_t n_tiles = cdiv(cdiv(nb, gemm_tile_rows()), mc);  // row-tile groups
    for (int64_t v0 = 0, band_i = 0; v0 < pb.V; v0 += Vc, ++band_i) {
      const int64_t vc = (pb.V - v0 < Vc) ? pb.V - v0 : Vc;
      const int64_t vt = cdiv(vc, kBN);

      WalkParams wg{};
      wg.total_tiles = int(n_tiles * vt);
      wg.tiles_minor = int(vt);
      if (FLCE_GRAD_SLICE_BYTES > 0) {
        // parts of the band whose W slice (D x 256 columns x 2 bytes a tile) fits the budget
        const int64_t parts = cdiv(pb.D * int64_t(kBN) * 2 * vt, FLCE_GRAD_SLICE_BYTES);
        wg.minor_part = parts > 1 ? int(cdiv(vt, parts)) : 0;
      }
      wg.num_kb = int(cdiv(pb.D, kBK));
      wg.b_row_off = int(v0);
      wg.dyn_mode = DYN_ROW_GROUPS;
      wg.dyn_rows = dyn;
      GradEpiParams ge{};
      ge.coef = coef_rows;
      ge.bval = bval;
      ge.N = int(nb);
      ge.V = int(pb.V);
      ge.chunk_v0 = int(v0);
      ge.err = err;
      if (ext) {
        ge.bias = opt->bias;
        ge.cw = cw;
        ge.softcap = opt->softcap;
      }
      FLCE_CUDA_CHECK(launch_grad_gemm(tmXk, tmWg, tmG, wg, ge, ext, pb.w_vd, pb.f16, stream));

      if (opt && opt->dbias) {
        ColsumParams cp{};
        cp.band = static_cast<const uint16_t*>(band);
        cp.N = int(nb);
        cp.ld = int(Vc);
        cp.cols = int(vc);
        cp.row_chunks = kColsumChunks;
        cp.partial = reinterpret_cast<float*>(ws + L.colsum);
        cp.out = opt->dbias + v0;
        cp.accumulate = (n0 > 0 || add_grads) ? 1 : 0;
        cp.f16 = pb.f16 ? 1 : 0;
        cp.scale = pb.f16 ? gval : nullptr;
        cp.scale_mul = 1.f / kF16GradScale;
        cp.dyn_rows = dyn;
        FLCE_CUDA_CHECK(launch_colsum(cp, stream));
      }

      // dW = X^T G (K = rows of the band); later row bands add into dW. With vocabulary
      // rows the GEMM computes G^T X instead (the operands swap): stored as it is into a
      // [V, D] dW, transposed into a [D, V] one.
      WalkParams ww{};
      ww.num_kb = int(cdiv(nb, kBK));
      ww.dyn_mode = DYN_K_ROWS;
      ww.dyn_rows = dyn;
      StoreEpiParams sw{(n0 > 0 || add_grads) ? 1 : 0, 0, err, 0, out_scale, 1.f / kF16GradScale};
      if (!dw_vocab_rows(pb.D, pb.w_vd)) {
        ww.total_tiles = int(vt * d_tiles_m);
        ww.tiles_minor = int(d_tiles_m);
        ww.col_major = 1;
        ww.minor_part = (FLCE_DW_MINOR_SPLIT > 1 && d_tiles_m % FLCE_DW_MINOR_SPLIT == 0)
                            ? int(d_tiles_m / FLCE_DW_MINOR_SPLIT) : 0;
        sw.x_off = int(v0);
        FLCE_CUDA_CHECK(launch_dw_gemm(tmXmn, tmGmn, tmDW, ww, sw, false, pb.f16, stream));
      } else {
        const int64_t v_groups = cdiv(cdiv(vc, gemm_tile_rows()), mc);
        ww.total_tiles = int(v_groups * d_tiles_n);
        ww.tiles_minor = int(d_tiles_n);
        ww.col_major = 0;
        if (pb.w_vd) {
          sw.y_off = int(v0);
          FLCE_CUDA_CHECK(launch_dw_gemm(tmGmn, tmXmn, tmDW, ww, sw, false, pb.f16, stream));
        } else {
          sw.x_off = int(v0);  // the tile's vocabulary rows land on dW columns v0 + ...
          FLCE_CUDA_CHECK(launch_dw_gemm(tmGmn, tmXmn, tmDWt, ww, sw, true, pb.f16, stream));
        }
      }

      WalkParams wx{};
      wx.total_tiles = int(n_tiles * d_tiles_n);
      wx.tiles_minor = int(d_tiles_n);
      wx.num_kb = int(cdiv(vc, kBK));
      wx.b_k0 = int(v0);
      wx.dyn_mode = DYN_ROW_GROUPS;
      wx.dyn_rows = dyn;
      if (FLCE_DX_SLICE_BYTES > 0) {
        // parts of D's tiles whose slice of the band's W (256 rows x vc x 2 bytes a tile) fits
        const int64_t parts = cdiv(int64_t(kBN) * vc * 2 * d_tiles_n, FLCE_DX_SLICE_BYTES);
        wx.minor_part = parts > 1 ? int(cdiv(d_tiles_n, parts)) : 0;
      }
      StoreEpiParams sx{band_i > 0 ? 1 : 0, 0, err, 0, out_scale, 1.f / kF16GradScale};
      FLCE_CUDA_CHECK(launch_dx_gemm(tmG, tmWx, tmDX, wx, sx, pb.w_vd, pb.f16, stream));
    }
    if (compact) {
      const ScatterCastParams sc{dx_acc, dXrows, slot, int(nb), int(pb.D), pb.f16 ? 1 : 0, err};
      FLCE_CUDA_CHECK(launch_scatter_cast(sc, sms, stream));
    } else if (!f32_out) {
      void* dXb = static_cast<uint8_t*>(dX) + size_t(n0) * size_t(pb.D) * 2;
      FLCE_CUDA_CHECK(launch_cast_16bit(dx_acc, dXb, size_t(nb) * size_t(pb.D), pb.f16, sms, err, stream));
    }
  }
  return FLCE_OK;
}

flce_status check_forward_outputs(const float* loss, const float* lse) {
  if (!loss || !lse) return FLCE_ERR_INVALID_ARG;
  if (!aligned(loss, 4) || !aligned(lse, 4)) return FLCE_ERR_ALIGNMENT;
  return FLCE_OK;
}

flce_status check_backward_outputs(const Problem& pb, const flce_options* opt, const float* lse,
                                   const float* grad_out, const void* dX, const float* dW) {
  const bool f32 = opt && opt->dX_f32;
  if (!lse || !grad_out || (!dX && !f32) || !dW) return FLCE_ERR_INVALID_ARG;
  if (pb.red == FLCE_REDUCTION_NONE) return FLCE_ERR_REDUCTION_NONE_GRAD;
  if (!aligned(lse, 4) || !aligned(grad_out, 4) || (!f32 && !aligned(dX, 16)) || !aligned(dW, 16))
    return FLCE_ERR_ALIGNMENT;
  return FLCE_OK;
}

}  // namespace

extern "C" {

flce_status flce_forward_ex(const void* X, const void* W, const int32_t* targets, int64_t N, int64_t D, int64_t V,
                            int32_t ignore_index, float label_smoothing, float zloss_scale, flce_reduction red,
                            const flce_options* opt, float* loss, float* lse, void* workspace, size_t ws_bytes,
                            struct CUstream_st* stream) {
  flce_status st = check_common(X, W, targets, N, D, V, label_smoothing, zloss_scale, int(red), workspace);
  if (st != FLCE_OK) return st;
  const Problem pb{X,   W, targets, N, D, V, ignore_index, label_smoothing, zloss_scale, red, opt_w_vd(opt),
                   opt_f16(opt)};
  if ((st = check_forward_outputs(loss, lse)) != FLCE_OK) return st;
  if ((st = check_options(opt, pb, false)) != FLCE_OK) return st;
  if (ws_bytes < fwd_layout(N, V).total) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  int sms = 0, dev = -1;
  if ((st = current_device(&sms, &dev)) != FLCE_OK) return st;
  if ((st = check_device_memory(dev, {{"X", X}, {"W", W}, {"targets", targets}, {"workspace", workspace},
                                      {"loss", loss}, {"lse", lse}})) != FLCE_OK ||
      (st = check_option_memory(dev, opt)) != FLCE_OK)
    return st;
  const int units = forward_max_units();
  if (units <= 0) {
    note_error("forward_max_units", "no resident cluster");
    return FLCE_ERR_CUDA;
  }
  return run_forward(pb, opt, FIN_LOSS, 0, loss, lse, nullptr, static_cast<uint8_t*>(workspace), ws_bytes, true,
                     sms, reinterpret_cast<cudaStream_t>(stream));
}

flce_status flce_forward(const void* X, const void* W, const int32_t* targets, int64_t N, int64_t D, int64_t V,
                         int32_t ignore_index, float label_smoothing, float zloss_scale, flce_reduction red,
                         float* loss, float* lse, void* workspace, size_t ws_bytes, struct CUstream_st* stream) {
  return flce_forward_ex(X, W, targets, N, D, V, ignore_index, label_smoothing, zloss_scale, red, nullptr, loss,
                         lse, workspace, ws_bytes, stream);
}

flce_status flce_backward_ex(const void* X, const void* W, const int32_t* targets, const float* lse, int64_t N,
                             int64_t D, int64_t V, int32_t ignore_index, float label_smoothing, float zloss_scale,
                             flce_reduction red, const flce_options* opt, const float* grad_out, void* dX, float* dW,
                             void* workspace, size_t ws_bytes, struct CUstream_st* stream) {
  flce_status st = check_common(X, W, targets, N, D, V, label_smoothing, zloss_scale, int(red), workspace);
  if (st != FLCE_OK) return st;
  const Problem pb{X,   W, targets, N, D, V, ignore_index, label_smoothing, zloss_scale, red, opt_w_vd(opt),
                   opt_f16(opt)};
  if ((st = check_backward_outputs(pb, opt, lse, grad_out, dX, dW)) != FLCE_OK) return st;
  if ((st = check_options(opt, pb, true)) != FLCE_OK) return st;
  if (ws_bytes < bwd_layout(backward_rows(opt, N), D, V).total) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  int sms = 0, dev = -1;
  if ((st = current_device(&sms, &dev)) != FLCE_OK) return st;
  if ((st = check_device_memory(dev, {{"X", X}, {"W", W}, {"targets", targets}, {"workspace", workspace},
                                      {"lse", lse}, {"grad_out", grad_out}, {"dX", dX}, {"dW", dW}})) != FLCE_OK ||
      (st = check_option_memory(dev, opt)) != FLCE_OK)
    return st;
  return run_backward(pb, opt, lse, grad_out, dX, dW, static_cast<uint8_t*>(workspace), true, sms,
                      reinterpret_cast<cudaStream_t>(stream));
}

flce_status flce_backward(const void* X, const void* W, const int32_t* targets, const float* lse, int64_t N,
                          int64_t D, int64_t V, int32_t ignore_index, float label_smoothing, float zloss_scale,
                          flce_reduction red, const float* grad_out, void* dX, float* dW, void* workspace,
                          size_t ws_bytes, struct CUstream_st* stream) {
  return flce_backward_ex(X, W, targets, lse, N, D, V, ignore_index, label_smoothing, zloss_scale, red, nullptr,
                          grad_out, dX, dW, workspace, ws_bytes, stream);
}

flce_status flce_forward_backward(const void* X, const void* W, const int32_t* targets, int64_t N, int64_t D,
                                  int64_t V, int32_t ignore_index, float label_smoothing, float zloss_scale,
                                  flce_reduction red, const flce_options* opt, const float* grad_out, float* loss,
                                  float* lse, void* dX, float* dW, void* workspace, size_t ws_bytes,
                                  struct CUstream_st* stream) {
  flce_status st = check_common(X, W, targets, N, D, V, label_smoothing, zloss_scale, int(red), workspace);
  if (st != FLCE_OK) return st;
  const Problem pb{X,   W, targets, N, D, V, ignore_index, label_smoothing, zloss_scale, red, opt_w_vd(opt),
                   opt_f16(opt)};
  if ((st = check_forward_outputs(loss, lse)) != FLCE_OK) return st;
  if ((st = check_backward_outputs(pb, opt, lse, grad_out, dX, dW)) != FLCE_OK) return st;
  if ((st = check_options(opt, pb, false)) != FLCE_OK) return st;
  {
    const size_t f = fwd_layout(N, V).total, b = bwd_layout(backward_rows(opt, N), D, V).total;
    if (ws_bytes < (f > b ? f : b)) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  }
  int sms = 0, dev = -1;
  if ((st = current_device(&sms, &dev)) != FLCE_OK) return st;
  if ((st = check_device_memory(dev, {{"X", X}, {"W", W}, {"targets", targets}, {"workspace", workspace},
                                      {"grad_out", grad_out}, {"loss", loss}, {"lse", lse}, {"dX", dX},
                                      {"dW", dW}})) != FLCE_OK ||
      (st = check_option_memory(dev, opt)) != FLCE_OK)
    return st;
  const int units = forward_max_units();
  if (units <= 0) {
    note_error("forward_max_units", "no resident cluster");
    return FLCE_ERR_CUDA;
  }
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if ((st = run_forward(pb, opt, FIN_LOSS, 0, loss, lse, nullptr, ws, ws_bytes, true, sms, s)) != FLCE_OK) return st;
  return run_backward(pb, opt, lse, grad_out, dX, dW, ws, false, sms, s);
}

flce_status flce_shard_stats(const void* X, const void* W, const int32_t* targets, int64_t N, int64_t D, int64_t V,
                             int64_t v_offset, int32_t ignore_index, float* stats, void* workspace, size_t ws_bytes,
                             struct CUstream_st* stream) {
  return flce_shard_stats_ex(X, W, targets, N, D, V, v_offset, ignore_index, nullptr, stats, workspace, ws_bytes,
                             stream);
}

flce_status flce_shard_stats_ex(const void* X, const void* W, const int32_t* targets, int64_t N, int64_t D,
                                int64_t V, int64_t v_offset, int32_t ignore_index, const flce_options* opt,
                                float* stats, void* workspace, size_t ws_bytes, struct CUstream_st* stream) {
  if (opt) {
    // only the storage options apply to shard statistics
    if (opt->softcap != 0.f || opt->bias || opt->class_weight || opt->predicted || opt->accuracy || opt->dbias ||
        opt->dX_f32 || opt->v_offset != 0 || opt->v_total != 0 || opt->row_band != 0 || opt->accumulate_grads)
      return FLCE_ERR_INVALID_ARG;
    if (opt->weight_layout != FLCE_WEIGHT_DV && opt->weight_layout != FLCE_WEIGHT_VD) return FLCE_ERR_INVALID_ARG;
    if (opt->input_dtype != FLCE_INPUT_BF16 && opt->input_dtype != FLCE_INPUT_F16) return FLCE_ERR_INVALID_ARG;
  }
  flce_status st = check_common(X, W, targets, N, D, V, 0.f, 0.f, 0, workspace);
  if (st != FLCE_OK) return st;
  if (!stats) return FLCE_ERR_INVALID_ARG;
  if (!aligned(stats, 4)) return FLCE_ERR_ALIGNMENT;
  if (v_offset < 0) return FLCE_ERR_INVALID_ARG;
  if (v_offset + V >= (int64_t(1) << 30)) return FLCE_ERR_TOO_LARGE;
  if (ws_bytes < fwd_layout(N, V).total) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  int sms = 0, dev = -1;
  if ((st = current_device(&sms, &dev)) != FLCE_OK) return st;
  if ((st = check_device_memory(dev, {{"X", X}, {"W", W}, {"targets", targets}, {"workspace", workspace},
                                      {"stats", stats}})) != FLCE_OK)
    return st;
  const int units = forward_max_units();
  if (units <= 0) {
    note_error("forward_max_units", "no resident cluster");
    return FLCE_ERR_CUDA;
  }
  const Problem pb{X, W, targets, N, D, V, ignore_index, 0.f, 0.f, FLCE_REDUCTION_SUM, opt_w_vd(opt), opt_f16(opt)};
  return run_forward(pb, nullptr, FIN_SHARD_STATS, v_offset, nullptr, nullptr, stats,
                     static_cast<uint8_t*>(workspace), ws_bytes, true, sms, reinterpret_cast<cudaStream_t>(stream));
}

flce_status flce_combine_shards(const float* stats, int32_t K, const int32_t* targets, int64_t N, int64_t v_total,
                                int32_t ignore_index, float label_smoothing, float zloss_scale, flce_reduction red,
                                float* loss, float* lse, void* workspace, size_t ws_bytes,
                                struct CUstream_st* stream) {
  if (!stats || !targets || !workspace || K < 1 || N < 1 || v_total < 1) return FLCE_ERR_INVALID_ARG;
  if (!(label_smoothing >= 0.f && label_smoothing < 1.f) || !(zloss_scale >= 0.f) || std::isinf(zloss_scale) ||
      int(red) < 0 || int(red) > 2)
    return FLCE_ERR_INVALID_ARG;
  if (N >= (int64_t(1) << 30) || v_total >= (int64_t(1) << 30) || K > 4096) return FLCE_ERR_TOO_LARGE;
  flce_status st = check_forward_outputs(loss, lse);
  if (st != FLCE_OK) return st;
  if (!aligned(stats, 4) || !aligned(targets, 4) || !aligned(workspace, 16)) return FLCE_ERR_ALIGNMENT;
  const FwdLayout L = fwd_layout(N, 8);
  if (ws_bytes < L.total) return FLCE_ERR_WORKSPACE_TOO_SMALL;
  int sms = 0, dev = -1;
  if ((st = current_device(&sms, &dev)) != FLCE_OK) return st;
  if ((st = check_device_memory(dev, {{"stats", stats}, {"targets", targets}, {"workspace", workspace},
                                      {"loss", loss}, {"lse", lse}})) != FLCE_OK)
    return st;
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  FLCE_CUDA_CHECK(cudaMemsetAsync(ws, 0, kHeaderBytes, s));
  FinalizeParams f{};
  f.mode = FIN_COMBINE;
  f.stats = stats;
  f.targets = targets;
  f.N = int(N);
  f.V = int(v_total);
  f.S = K;
  f.ignore_index = ignore_index;
  f.eps = label_smoothing;
  f.zscale = zloss_scale;
  f.reduction = int(red);
  f.lse = lse;
  f.loss = loss;
  f.block_sum = reinterpret_cast<double*>(ws + L.block_sum);
  f.block_wsum = reinterpret_cast<double*>(ws + L.block_wsum);
  f.block_cnt = reinterpret_cast<int*>(ws + L.block_cnt);
  f.block_correct = reinterpret_cast<int*>(ws + L.block_correct);
  f.err = reinterpret_cast<int*>(ws + kHdrErr);
  FLCE_CUDA_CHECK(launch_finalize(f, L.blocks, s));
  return FLCE_OK;
}

int64_t flce_backward_band_width(int64_t N, int64_t D, int64_t V, const flce_options* opt) {
  if (!sizes_ok(N, D, V) || !sizes_in_range(N, D, V)) return 0;
  int sms = 0;
  if (current_device(&sms) != FLCE_OK) return 0;
  const int64_t rows = backward_rows(opt, N);
  const BwdLayout L = bwd_layout(rows, D, V);
  return pick_band_width(L.Vc, rows, D, V, opt_w_vd(opt), walk_max_clusters());
}

flce_status flce_check_device_error(void* workspace, struct CUstream_st* stream_) {
  if (!workspace) return FLCE_ERR_INVALID_ARG;
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  int word = 0;
  FLCE_CUDA_CHECK(cudaStreamSynchronize(stream));
  FLCE_CUDA_CHECK(cudaMemcpy(&word, workspace, sizeof(int), cudaMemcpyDeviceToHost));
  FLCE_CUDA_CHECK(cudaMemset(workspace, 0, sizeof(int)));
  if (word & FLCE_DEVERR_TIMEOUT) return FLCE_ERR_TIMEOUT;
  if (word & FLCE_DEVERR_BAD_TARGET) return FLCE_ERR_BAD_TARGET;
  if (word & FLCE_DEVERR_F16_RANGE) return FLCE_ERR_F16_RANGE;
  return FLCE_OK;
}

}  // extern "C"
