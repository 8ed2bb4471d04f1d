// gmm_kernels.cuh -- device-side data shared by the EM-step kernels and the
// host planner: the per-call scalars and the fused kernel's argument block.
#pragma once
#include <cstdint>

#include "layout.cuh"

namespace gmm {

constexpr int kMaxD = 128;

// Scale of the fp16 responsibility operand: r is stored as r * kRScale, so
// that responsibilities down to 2^-24 / kRScale stay out of the fp16
// subnormal range (FAST, one piece: 2^10; PRECISE, hi + lo pieces: 2^15).
template <int NP>
__host__ __device__ constexpr float kRScale() { return NP == 1 ? 1024.f : 32768.f; }

// Device status bits (or-ed into a word in global memory).
enum : uint32_t {
  ST_TIMEOUT = 1u,
  ST_NONFINITE = 2u,
  ST_RANGE = 4u,
  ST_CAPACITY = 8u,       // threshold assignment: more entries than the output holds
};

// Per-call scalars computed on the device before the main pass.
struct Meta {
  float shift[kMaxD];     // data are used as x' = (x - shift) * scale
  float scale;            // power of two
  float inv_scale;
  uint32_t absmax_bits;   // max |x| over X (float bits; written by the scan)
  uint32_t bmax_bits;     // FAST: max over components and features of |mu'/s2'|, |1/(2 s2')| (log2 units)
  float pscale;           // FAST: the one power-of-two scale of every parameter row
  float pinv;             // 1 / pscale
};

enum KernelId : int {
  K_ABSMAX, K_ABSMAX_VEC, K_META, K_PARAMS_FAST, K_PARAMS_PRECISE,
  K_FUSED_1_1_2, K_FUSED_1_2_2, K_FUSED_2_1_1, K_LSE_COMBINE, K_FINALIZE,
  K_TOPM_COMBINE, K_LL_TOTAL, K_TOPM_1_1_2, K_TOPM_1_2_2, K_TOPM_2_1_1,
  K_THRESH_COUNT, K_THRESH_SCAN, K_THRESH_SCATTER,
  K_TIED_PREP, K_GRAM_REDUCE, K_SIGMA_TIED,
  K_BMAX, K_FUSED_2_2_1, K_TOPM_2_2_1, K_TIED_INV,
};

// The tied model's Gram matrix on the tensor cores (gram.cu): kernel handle for
// np operand pieces, nch atom columns and bf16 or f32 data; its dynamic shared
// memory and threads per CTA.  Launch: two CTAs per SM (at most one per tile),
// arguments (FusedArgs, double* partials [CTA][D][D]).
const void* gram_handle(int np, int nch, bool xb);
size_t gram_smem(int np, int nch);
int gram_threads();

// Handles of the two-team FAST kernels (em_fast.cu), nch = 1 or 2, one per
// mode (MODE_LSE, MODE_GIVEN, MODE_TOPM with candidate lists of maxm = 2, 4
// or 8; NULL for MODE_EM, which runs on the fused kernel), and their dynamic
// shared-memory size (512 threads per CTA).
const void* emfast_handle(int nch, int mode, int maxm = 0);
size_t emfast_smem(int nch);
constexpr int kEmFastThreads = 512;

// Threshold assignment: points per block of the count and scatter kernels.
constexpr int kThreshBlock = 256;

// Approximate top-k EM (topk_em.cu): pairs per chunk of the statistics
// kernel and the kernels.  Launch shapes: COUNT and FILL one CTA of 32 threads
// per tile of points with K * 4 bytes of dynamic shared memory; SCAN one CTA
// of 1024 per 32 components; BASE one
// CTA of 1024; STATS / STATS_VEC one CTA of 128 per chunk (chunks beyond the
// device-side total return at once; partials of 3 D + 1 doubles per chunk;
// STATS_VEC for rows of a multiple of 16 bytes); FINAL one CTA of 128 per
// component.
constexpr int kTkChunk = 2048;
enum TopkKernel : int { TK_COUNT, TK_SCAN, TK_BASE, TK_FILL, TK_STATS, TK_STATS_VEC, TK_FINAL };
const void* topk_handle(TopkKernel id, bool xb);

// topm_refine.cu: direct-form recomputation of the top-m candidates' logits
// (per-component rows (mu, 1/s2) padded to kMaxD features and constants, then
// eight lanes per point; vec: X read as feature pairs; maxm 2/4/8/16).
const void* refine_params_handle();
const void* refine_handle(bool xb, bool vec, int maxm);

// Host-side handle of a kernel, for cudaLaunchKernelEx (argument order and
// types as in gmm_kernels.cu).
const void* kernel_handle(KernelId id);

enum Mode : int {
  MODE_EM = 0,      // logits, normaliser across the cluster, statistics
  MODE_LSE = 1,     // logits, normaliser across the cluster, write it out
  MODE_GIVEN = 2,   // logits, normaliser read from memory, statistics
  MODE_TOPM = 3,    // logits, normaliser and top-m across the cluster
};

struct FusedArgs {
  const void* X;
  int64_t N;
  int D;
  int K;
  int K_pad;           // K rounded up to the slice size
  int x_bf16;
  int mode;
  int C;               // CTAs per cluster (slices sharing one point tile)
  int n_tiles;         // ceil(N / 128)
  int flush_tiles;     // statistics leave tensor memory every this many tiles
  int F;               // doubles per component row of the partial statistics
  int topm;            // m of the top-m mode
  int topm_max;        // m rounded up to a power of two (2..16): candidate list length
  const uint8_t* p_img;   // parameter operand images, one per slice
  const uint8_t* c_img;   // FAST: the logit constants as a 128 x 16 operand, one per slice
  const float* cadj;      // per-component logit constant (log2 units)
  const float* iscale;    // per-component scale of the logit accumulator
  const Meta* meta;
  double* part;           // partial statistics [tile group][K_pad][F]
  double* ll_part;        // per tile group log-likelihood partials
  float* lse_part;        // MODE_LSE output [K group][N] (log2 units)
  const float* lse_in;    // MODE_GIVEN input [N] (log2 units)
  float* topm_val;        // MODE_TOPM output: responsibilities [N][m] (one K group), or
                          // per-group log2 logits [K group][N][m] (several K groups)
  int32_t* topm_idx;      // MODE_TOPM output component indices, same layout
  int topm_groups;        // number of K groups (gridDim.y); 1: final output
  uint32_t* status;
  uint32_t max_polls;     // polls per bounded wait (0: the default)
};

struct Small {
  float cadj[kSlice];
  float iscale[kSlice];
  float pair_m[2][kBN];
  float pair_s[2][kBN];
  float xrecv[2][8][kBN];  // row normalisers pushed by each CTA of the cluster, per slot
  float lse_row[kBN];     // MODE_TOPM: normaliser of each row of the tile (log2 units)
  double ll_red[8];
  uint64_t full_a[2];
  uint64_t empty_g[2][8];  // per stage: 16-row group g no longer read by the MMAs
  uint64_t p_full;
  uint64_t pfull[3];       // streamed parameter image: ring slot filled
  uint64_t pempty[3];      // streamed parameter image: ring slot read by its MMAs
  uint64_t acc1_full;
  uint64_t acc1_empty;
  uint64_t r_full[4];     // lane quarter q's rows written to R slot q & 1 (64 threads), one phase per tile
  uint64_t r_done[4];     // lane quarter q's rows read by the statistics MMA
  uint64_t acc2_full;
  uint64_t acc2_empty;
  uint64_t xready[2];     // slot filled: every CTA of the cluster has pushed its row normalisers
  uint64_t tready;        // MODE_TOPM: candidate lists of every CTA of the cluster written
  uint64_t tfree;         // MODE_TOPM: candidate lists of every CTA of the cluster consumed
  uint64_t drain;
  uint32_t tmem_base;
  uint32_t abort_flag;
  uint32_t poll_limit;     // follows abort_flag (read by the bounded waits)
};

// Shared-memory plan of the fused kernel for NP operand pieces (1: fp16,
// 2: fp16 hi/lo), NCH 64-feature atom columns per data part, NST data stages:
//   [data stages | parameter image (or its ring) | Small | R tile | ones]
// MODE_TOPM runs with one data stage; the second stage (or, with a single
// stage, the R tile area) holds the per-row candidate lists.
template <int NP, int NCH, int NST>
struct Cfg {
  static constexpr int kPieceBytes = 2 * NCH * kChunkBytes;          // [x | x^2] for 128 rows
  static constexpr int kStageBytes = NP * kPieceBytes;
  static constexpr int kOffA = 0;
  static constexpr int kOffP = NST * kStageBytes;
  // Two pieces of 128 features (PRECISE, D > 64): the 128 KB parameter image
  // does not fit beside the 128 KB data stage, so it streams through a ring
  // of kPRing 16 KB chunks, read again (from L2) for every tile.
  static constexpr bool kStreamP = NP == 2 && NCH == 2;
  static constexpr int kPRing = 3;
  static constexpr int kParamBytes = kStreamP ? kPRing * kChunkBytes : NP * kPieceBytes;
  static constexpr int kOffSmall = kOffP + kParamBytes;
  static constexpr int kOffR = (kOffSmall + static_cast<int>(sizeof(Small)) + 1023) / 1024 * 1024;
  static constexpr int kRBytes = 2 * kRSlotBytes * 2;                // 2 slots x 32 points x 128 comps x 16 bit
  static constexpr int kOffOnes = kOffR + NP * kRBytes;             // 16 x 64 fp16 ones
  static constexpr int kEnd = kOffOnes + 2048;
  static constexpr int kDp = NCH * kAtomElems;
  static constexpr int kF2 = 2 * kDp + 16;                            // statistics columns in TMEM
  static constexpr uint32_t kAcc1Col = 0;
  static constexpr uint32_t kAcc2Col = 128;
  static constexpr int kThreads = 13 * 32;
};

// MODE_TOPM candidate lists: for each of the 128 rows of a tile and each of
// the two column halves, the MAXM best (logit, component) pairs (at most
// 24 KB, within one data stage or the R tile area of every configuration).
__host__ __device__ constexpr int topm_list_bytes(int maxm) { return kBN * 2 * maxm * 6; }

}  // namespace gmm
