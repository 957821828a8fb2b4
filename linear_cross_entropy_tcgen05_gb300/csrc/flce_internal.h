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

// Output tiles of the tensor-core GEMMs: 128 rows per CTA (TMEM lanes) x 256 columns,
// a CTA pair (cluster of 2) owning 256 x 256; K staged 64 bf16 (128 bytes, one
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
// triples per row.
constexpr int kMaxSplits = 64;

// Tile walk of the non-forward GEMMs; see the kernel for how a tile index maps to
// operand rows.
enum WalkKind : int { WALK_GRAD = 0, WALK_DW = 1, WALK_DX = 2 };

struct WalkParams {
  int total_tiles;   // tiles in this launch
  int tiles_minor;   // tiles along the fast-varying output dimension
  int num_kb;        // 64-wide K blocks per tile
  int a_k0, b_k0;    // K coordinate of the first block (A, B)
  int b_row_off;     // added to the B operand's row/column coordinate
};

struct FwdParams {
  const int32_t* targets;
  int N, V;
  int n_tiles, v_tiles;
  int gN, S;       // grid = gN row tiles x S vocabulary ranges (CTA pairs)
  int num_kb;      // K blocks over D
  int want_sum_z;  // label smoothing needs sum_j z_ij
  float* part_m;   // [S][N] running max
  float* part_d;   // [S][N] sum of exp(z - max)
  float* part_s;   // [S][N] sum of z
  float* tgt;      // [N] target logit
  int* err;
};

struct GradEpiParams {
  const float4* coef;  // per row {a, -lse*log2e, b, bits(target or -1)}
  const float* cval;   // device scalar: g (1 - eps), subtracted at the target column
  int N, V;
  int chunk_v0;        // first vocabulary column of the current band
  int* err;
};

struct StoreEpiParams {
  int reduce_add;  // 0: store, 1: element-wise add into the destination
  int x_off;       // added to the B-row coordinate to form the destination column
  int* err;
};

struct FinalizeParams {
  const float* part_m;
  const float* part_d;
  const float* part_s;
  const float* tgt;
  const int32_t* targets;
  int N, V, S;
  int ignore_index;
  float eps, zscale;
  int reduction;        // 0 mean, 1 sum, 2 none
  float* lse;
  float* loss;          // [1] or [N]
  double* block_sum;    // [blocks]
  int* block_cnt;       // [blocks]
  int* err;
};

struct PrepParams {
  const int32_t* targets;
  const float* lse;
  const float* grad_out;
  int N, V;
  int ignore_index;
  float eps, zscale;
  int reduction;
  float4* coef;
  float* cval;
  int* err;
};

// Rows of one GEMM output tile (a CTA pair: 2 x 128).
int gemm_tile_rows();
// Rows (K-major) or columns (MN-major) of the B operand each CTA loads: 256 / pair size.
int gemm_b_rows_per_cta();
// CTA pairs of the forward GEMM that can be resident at once on the current device.
int forward_max_units();

cudaError_t launch_forward_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const FwdParams& p,
                                cudaStream_t stream);
cudaError_t launch_finalize(const FinalizeParams& p, int blocks, cudaStream_t stream);
cudaError_t launch_prep(const PrepParams& p, cudaStream_t stream);
// The walk GEMMs size their own grids: min(tiles, resident CTA pairs) clusters of 2.
cudaError_t launch_grad_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                             const WalkParams& w, const GradEpiParams& e, cudaStream_t stream);
cudaError_t launch_dw_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                           const WalkParams& w, const StoreEpiParams& e, cudaStream_t stream);
cudaError_t launch_dx_gemm(const CUtensorMap& tmA, const CUtensorMap& tmB, const CUtensorMap& tmC,
                           const WalkParams& w, const StoreEpiParams& e, cudaStream_t stream);
cudaError_t launch_cast_bf16(const float* src, void* dst, size_t n, int num_sms, cudaStream_t stream);

constexpr int kFinalizeThreads = 256;

}  // namespace flce
