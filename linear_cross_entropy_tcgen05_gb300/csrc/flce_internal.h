// flce_internal.h -- parameter blocks and launchers shared by the host API and the
// kernels of the fused linear cross-entropy library. Not part of the public ABI.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace flce {

// Device error bits kept in the first word of the workspace (mapped to flce_status
// values by flce_check_device_error).
constexpr int FLCE_DEVERR_BAD_TARGET = 1;
constexpr int FLCE_DEVERR_TIMEOUT = 2;
constexpr int FLCE_DEVERR_F16_RANGE = 4;  // a scaled f16 gradient coefficient exceeds the f16 range

// Output tiles of the tensor-core GEMMs: 128 rows per CTA (TMEM lanes) x 256 columns,
// a CTA pair owning 256 x 256; K staged 64 16-bit elements (128 bytes, one
// 128B-swizzle row) at a time.
constexpr int kBM = 128;
constexpr int kBN = 256;
constexpr int kBK = 64;
constexpr int kThreads = 192;      // warp 0: TMA producer, warp 1: MMA issuer, warps 2-5: epilogue
constexpr int kEpiThreads = 128;
constexpr int kABytes = kBM * kBK * 2;          // 16 KB
constexpr int kStagingBytes = 128 * 128;        // one 128-row x 128-byte epilogue store box
constexpr int kBarrierBytes = 256;

// Forward split of the vocabulary: at most this many partial (max, sum-exp, sum-z)
// triples per row (one per vocabulary chunk of the forward's units).
#ifndef FLCE_FWD_MAX_SPLITS
#define FLCE_FWD_MAX_SPLITS 64
#endif
constexpr int kMaxSplits = FLCE_FWD_MAX_SPLITS;
// Forward: row tiles a CTA pair computes against each W tile before moving on.
#ifndef FLCE_FWD_ROW_BLOCK
#define FLCE_FWD_ROW_BLOCK 1
#endif
constexpr int kFwdRowBlock = FLCE_FWD_ROW_BLOCK;
// Forward: cluster row blocks per panel. The clusters working at one time take the
// blocks of one panel through neighbouring vocabulary chunks, so they share the panel's
// rows of X and the chunks' W tiles through L2. FLCE_FWD_PANEL > 0 fixes the count;
// 0 sizes the panel to FLCE_FWD_PANEL_BYTES of X (8 blocks at D = 4096).
#ifndef FLCE_FWD_PANEL
#define FLCE_FWD_PANEL 0
#endif
#ifndef FLCE_FWD_PANEL_BYTES
#define FLCE_FWD_PANEL_BYTES (int64_t(32) << 20)
#endif
// Diagnostic build: the GEMMs add the cycles their MMA thread waited for operands and
// for the epilogue, its total cycles, and the cycles their producer waited for free
// stages, to four uint64 counters at bytes 32 + 32 * (kind + 1) of the workspace header
// (kind: -1 forward, 0 gradient, 1 dW, 2 dX) (0: off).
#ifndef FLCE_WAIT_STATS
#define FLCE_WAIT_STATS 0
#endif
// CTA pairs per cluster: 2 makes two pairs share every B tile (one TMA multicast load
// instead of two), 1 gives every pair its own loads.
#ifndef FLCE_PAIRS_PER_CLUSTER
#define FLCE_PAIRS_PER_CLUSTER 2
#endif
// dW GEMM of a [D, V] dW: walk the D row groups in this many parts, each part across all
// vocabulary tiles of the band before the next, so a wave re-reads fewer columns of X.
#ifndef FLCE_DW_MINOR_SPLIT
#define FLCE_DW_MINOR_SPLIT 2
#endif
// Gradient GEMM: walk the band's vocabulary tiles in parts whose W slice is at most this
// many bytes, each part across all row groups before the next, so that the slice stays in
// the L2 share that data read from both dies can use (0: one part).
#ifndef FLCE_GRAD_SLICE_BYTES
#define FLCE_GRAD_SLICE_BYTES (int64_t(40) << 20)
#endif
// dX GEMM: the same for its D tiles (each reads a 256-row slice of the band's W); off by
// default (measured even: the G rows are then read once per part).
#ifndef FLCE_DX_SLICE_BYTES
#define FLCE_DX_SLICE_BYTES int64_t(0)
#endif
// L2 policies (0 normal, 1 evict-first, 2 evict-last) of the dX GEMM's A operand (the
// gradient band), the dW GEMM's operands, and the gradient GEMM's band store.
#ifndef FLCE_DX_A_POL
#define FLCE_DX_A_POL 0
#endif
#ifndef FLCE_DW_A_POL
#define FLCE_DW_A_POL 0
#endif
#ifndef FLCE_DW_B_POL
#define FLCE_DW_B_POL 0
#endif
#ifndef FLCE_GRAD_STORE_POL
#define FLCE_GRAD_STORE_POL 1
#endif
// L2 cache-policy hints on the GEMMs' TMA traffic (1: on).
#ifndef FLCE_L2_HINTS
#define FLCE_L2_HINTS 1
#endif

// Tile walk of the non-forward GEMMs; see the kernel for how a tile index maps to
// operand rows.
enum WalkKind : int { WALK_GRAD = 0, WALK_DW = 1, WALK_DX = 2 };

// A walk whose rows are the valid rows of the batch, compacted on the device, learns
// their count when it starts: dyn_rows points at it (written by an earlier kernel).
enum DynRows : int {
  DYN_NONE = 0,
  DYN_ROW_GROUPS = 1,  // row-tile groups (col_major == 0): only those holding valid rows
  DYN_K_ROWS = 2,      // K runs over rows: only the 64-row blocks holding valid rows
};

struct WalkParams {
  int total_tiles;   // tiles in this launch
  int tiles_minor;   // tiles along the fast-varying output dimension
  int num_kb;        // 64-wide K blocks per tile
  int a_k0, b_k0;    // K coordinate of the first block (A, B)
  int b_row_off;     // added to the B operand's row/column coordinate
  int col_major;     // 1: the slow index runs over output columns (all row tiles of a
                     // column in flight), 0: over row-tile groups
  int dyn_mode;          // DynRows: how *dyn_rows bounds the walk (at least one group or block)
  const int* dyn_rows;   // device count of valid rows, or null
  int minor_part;        // > 0: walk the minor tiles in parts of this many (the last part may
                         // be narrower), each part across all majors before the next; 0: off
};

// Rows past the valid-row count that the compacted operands hold as zeros (with an
// ignored-row coefficient), so that the last row-tile group and K block a walk touches
// read defined values: a multiple of every walk's row granularity (512 and 64).
constexpr int kCompactPadRows = 1024;

struct CompactParams {
  const int32_t* targets;
  int N;
  int ignore_index;
  int* rows;     // [N] original index of each valid row, in order
  int* slot;     // [N] compacted index of each row, -1 if ignored
  int* n_valid;  // device scalar
};

struct GatherParams {
  const void* X;         // 16-bit [N, D]
  void* Xc;              // 16-bit [N, D]: valid rows first, then zeros up to the padding
  const float4* coef;    // [N] per-row gradient coefficients, or null (the forward: none)
  float4* coef_c;        // [N] the same in compacted order, ignored-row values in the padding
  const int* rows;
  const int* n_valid;
  int N, D;
};

struct ScatterCastParams {
  const float* acc;   // fp32 [N, D], compacted rows
  void* dX;           // 16-bit [N, D], original rows (zero for ignored rows)
  const int* slot;
  int N, D;
  int f16;
  const int* err;     // the call's error word: a pipeline timeout makes every dX element NaN
};

// Sentinel target of an ignored row in the per-row gradient coefficients.
constexpr int kIgnoredRow = int(0x80000000);

struct FwdParams {
  const int32_t* targets;
  int N, V;
  int n_tiles, v_tiles;
  int n_blocks;     // cluster row blocks (MC pairs x kFwdRowBlock row tiles each)
  int panel;        // cluster row blocks per panel (at most; fewer if there are fewer blocks)
  int chunk_tiles;  // vocabulary tiles per chunk; one partial statistic per row and chunk
  int n_chunks;     // chunks over the vocabulary (at most kMaxSplits)
  int total_units;  // n_blocks x n_chunks units, handed out in order by a ticket counter
  int* ticket;      // the counter (zero when the launch starts)
  const int* dyn_rows;  // valid-row compaction: device count of the rows of X (the valid
                        // rows, gathered), which replaces N, n_tiles, n_blocks, total_units
  const int* row_of;    // valid-row compaction: original row of each compacted row, or null
  int num_kb;       // K blocks over D
  int want_sum_z;  // label smoothing needs sum_j z_ij
  int ignore_index;
  int y_offset;    // vocabulary shard: global index of W's first column
  float* part_m;   // [S][N] running max
  float* part_d;   // [S][N] sum of exp(z - max)
  float* part_s;   // [S][N] sum of z (sum of w_j u_j with class weights)
  float* tgt;      // [N] target logit
  int* err;
  // extended epilogue only
  const float* bias;  // [V] or null
  const float* cw;    // [V] class weights or null
  float softcap;      // 0: off
  int* part_idx;      // [S][N] first column of the range maximum, or null
};

struct GradEpiParams {
  const float4* coef;  // per row {A, -lse*log2e, C, target column in W (or kIgnoredRow)}
  const float* bval;   // device scalar B = g eps / V_total: G -= B w_j on valid rows
  int N, V;
  int chunk_v0;        // first vocabulary column of the current band
  int* err;
  // extended epilogue only
  const float* bias;  // [V] or null
  const float* cw;    // [V] or null
  float softcap;      // 0: off
};

struct StoreEpiParams {
  int reduce_add;      // 0: store, 1: element-wise add into the destination
  int x_off;           // added to the B-row coordinate to form the destination column
  int* err;
  int y_off;           // added to the A-row coordinate to form the destination row
  const float* scale;  // null, or the accumulator is multiplied by *scale * scale_mul
  float scale_mul;
};

// f16 inputs: the gradient band holds G * kF16GradScale / g (g = the loss scale of the
// gradient), so that probabilities near 1/V stay normal f16 numbers; the dW and dX
// epilogues multiply by g / kF16GradScale. |G / g| is at most (1 - eps) w_y +
// (eps / V) sum_j w_j + 2 s lse, which must stay below 65504 / kF16GradScale = 64.
constexpr float kF16GradScale = 1024.f;

enum FinalizeMode : int { FIN_LOSS = 0, FIN_SHARD_STATS = 1, FIN_COMBINE = 2 };

struct FinalizeParams {
  int mode;
  const float* part_m;  // FIN_LOSS / FIN_SHARD_STATS: [S][N] partials of the forward GEMM
  const float* part_d;
  const float* part_s;
  const float* tgt;
  const int* part_idx;  // [S][N] or null (argmax)
  const float* stats;   // FIN_COMBINE: [S][4][N] shard statistics (S = shard count)
  const int32_t* targets;
  int N, V, S;          // V: the full vocabulary (v_total)
  int V_local;          // FIN_SHARD_STATS: columns of this shard
  int v_offset;         // FIN_SHARD_STATS: global index of the shard's first column
  int ignore_index;
  float eps, zscale;
  int reduction;        // 0 mean, 1 sum, 2 none
  const float* cw;      // [V] class weights or null
  const float* wtot;    // device scalar sum_j w_j (with cw)
  float* lse;
  const int* slot;      // valid-row compaction of the forward: the partial statistics of row r
                        // sit at slot[r] (-1: an ignored row), or null (at r)
  float* loss;          // [1] or [N]
  float* stats_out;     // FIN_SHARD_STATS: [4][N]
  int* predicted;       // [N] or null
  float* accuracy;      // [1] or null
  double* block_sum;    // [blocks] loss partial sums
  double* block_wsum;   // [blocks] mean denominators (valid rows or their weights)
  int* block_cnt;       // [blocks] valid rows
  int* block_correct;   // [blocks] argmax hits
  int* err;
};

struct PrepParams {
  const int32_t* targets;
  const float* lse;
  const float* grad_out;
  int N;
  int V;                // full vocabulary (v_total)
  int y_offset;         // vocabulary shard: global index of W's first column
  int ignore_index;
  float eps, zscale;
  int reduction;
  const float* cw;      // [V] class weights or null
  const float* wtot;    // device scalar sum_j w_j (with cw)
  float4* coef;
  float* gval;          // device scalar g (written by the denominator pass)
  float* bval;          // device scalar B = g' eps / V
  float gscale;         // > 0: g' = gscale replaces g in B and the coefficients (f16 band)
  int* err;
};

struct ColsumParams {
  const uint16_t* band;  // bf16 or f16 [N][ld]
  int N, ld, cols;
  int row_chunks;
  float* partial;        // [row_chunks][cols]
  float* out;            // [cols]
  int accumulate;        // add to out instead of overwriting
  int f16;               // the band holds f16 values
  const float* scale;    // null, or column sums are multiplied by *scale * scale_mul
  float scale_mul;
  const int* dyn_rows;   // device count of the band's rows to sum (compacted valid rows), or null
};

// Rows of one GEMM output tile (a CTA pair: 2 x 128).
int gemm_tile_rows();
// CTA pairs per cluster (pairs of a cluster share B); walks count row tiles in these units.
int gemm_pairs_per_cluster();
// Rows (K-major) or columns (MN-major) of the B operand each CTA loads: 256 / pair size.
int gemm_b_rows_per_cta();
// CTA pairs of the forward GEMM that can be resident at once on the current device.
int forward_max_units();
// Clusters of the backward GEMMs that can be resident at once on the current device.
int walk_max_clusters();

// ext: the extended epilogue (bias, softcap, class weights, argmax); else the plain one.
// w_vd: W is stored [V, D] (B is K-major); else [D, V] (B is MN-major).
// f16: X and W are f16 (else bf16).
cudaError_t launch_forward_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const FwdParams& p, bool ext,
                                bool w_vd, bool f16, cudaStream_t stream);
cudaError_t launch_finalize(const FinalizeParams& p, int blocks, cudaStream_t stream);
// g and B from the mean denominator over all rows (one block).
cudaError_t launch_denominator(const PrepParams& p, cudaStream_t stream);
// Per-row gradient coefficients of rows [0, n_rows) of p.targets / p.lse into p.coef.
cudaError_t launch_coef(const PrepParams& p, int n_rows, cudaStream_t stream);
// One block whose pipeline wait times out on purpose (bounded): sets the timeout bit.
cudaError_t launch_wait_selftest(int* err, cudaStream_t stream);
// out[0] = sum of v[0..n) in a fixed order (one block).
cudaError_t launch_sum(const float* v, int n, float* out, cudaStream_t stream);
// Column sums of a bf16 band, fixed order (two kernels).
cudaError_t launch_colsum(const ColsumParams& p, cudaStream_t stream);
// The walk GEMMs size their own grids: min(tile groups, resident clusters) clusters.
// w_vd as in launch_forward_gemm: it sets the major-ness of W, the B operand of the
// gradient and dX GEMMs. The dW GEMM takes both operands MN-major in either layout (the
// caller swaps them to compute G^T X, rows = vocabulary tiles); transposed_store writes
// such G^T X tiles into a [D, V] dW through an unswizzled 128 x 32 box.
cudaError_t launch_grad_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                             const WalkParams& w, const GradEpiParams& e, bool ext, bool w_vd, bool f16,
                             cudaStream_t stream);
cudaError_t launch_dw_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                           const WalkParams& w, const StoreEpiParams& e, bool transposed_store, bool f16,
                           cudaStream_t stream);
cudaError_t launch_dx_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                           const WalkParams& w, const StoreEpiParams& e, bool w_vd, bool f16, cudaStream_t stream);
// fp32 -> bf16 (or f16) of n elements, n a multiple of 4.
cudaError_t launch_cast_16bit(const float* src, void* dst, size_t n, bool f16, int num_sms, const int* err,
                              cudaStream_t stream);
// Valid-row compaction of the backward: the list of valid rows and their count (one
// block), the gather of their X rows and coefficients, and the final cast of the
// compacted dX accumulator back to the original rows.
cudaError_t launch_compact_rows(const CompactParams& p, cudaStream_t stream);
cudaError_t launch_gather_rows(const GatherParams& p, int num_sms, cudaStream_t stream);
cudaError_t launch_scatter_cast(const ScatterCastParams& p, int num_sms, cudaStream_t stream);

constexpr int kFinalizeThreads = 256;

// Kernels this library has launched in the process (every launch site counts itself).
void count_launch();
unsigned long long launches_so_far();

// Diagnostic device timing of the GEMM launches (flce_profile_gemms / flce_profile_read):
// when enabled, every GEMM launch is bracketed by a pair of CUDA events on its stream.
enum GemmKind : int { GEMM_FORWARD = 0, GEMM_GRADIENT = 1, GEMM_DW = 2, GEMM_DX = 3, GEMM_KINDS = 4 };
void profile_begin(int kind, cudaStream_t stream);
void profile_end(int kind, cudaStream_t stream);
void profile_enable(bool on);
cudaError_t profile_read(double* ms, unsigned long long* launches);

}  // namespace flce
