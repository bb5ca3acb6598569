// Internal interface between the host planner (api.cpp) and the CUDA
// kernels.  Every kernel takes one __grid_constant__ parameter struct, so a
// launch needs no host-to-device descriptor copy.
#pragma once

#include <cuda.h>           // CUtensorMap (type only; the driver is reached at run time)
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace muon {

// ---- device status word bits ------------------------------------------------
constexpr unsigned kDevTimeout = 1u;
constexpr unsigned kDevNonfinite = 2u;
constexpr unsigned kDevBounds = 4u;   // debug builds: an index or TMA coordinate check failed

#ifdef __CUDACC__
// Debug builds (-DMUON_DEBUG): a failed check sets kDevBounds in the status
// word and the caller skips the access it guards (a skipped copy leaves its
// consumer to run into a bounded wait).  In release builds it is `true`.
__device__ __forceinline__ bool dbg_ok(bool ok, unsigned* status) {
#ifdef MUON_DEBUG
  if (!ok) atomicOr(status, kDevBounds);
  return ok;
#else
  (void)ok;
  (void)status;
  return true;
#endif
}
#endif

// ---- limits ------------------------------------------------------------------
constexpr int kMaxSlices = 64;    // user (group, batch-range) pieces per launch
constexpr int kMaxNsGroups = 12;  // core shapes per NS launch
constexpr int kMaxSteps = 64;

// ---- K1: momentum / norm / cast / transpose ---------------------------------
constexpr int kPrepTile = 64;     // 64 x 64 tile of the stored [r][c] matrix

struct PrepSlice {
  const void* G;          // [count][r][c] (gradient, or the NS input)
  float* Mom;             // [count][r][c] fp32 (step mode), else null
  __nv_bfloat16* direct;  // workspace Xt in [r][c] layout (rows > cols), else null
  __nv_bfloat16* transp;  // workspace Xt in [c][r] layout (rows <= cols), else null
  __nv_bfloat16* direct_lo;   // high-precision mode: lo = bf16(D - hi) beside each, else null
  __nv_bfloat16* transp_lo;
  float* ssq_part;        // [count][tiles] per-tile partial sum of squares
  float* inv;             // [count] 1/(||D||_F + eps)
  unsigned* cnt;          // [count] arrival counters (left at zero)
  int64_t r, c;
  int64_t pitch_d, pitch_t;   // row pitches (elements)
  int64_t mstride_d, mstride_t;
  int count;
  int g_dtype;            // 0 f32, 1 bf16
  int tiles_r, tiles_c;
  int tile_base;          // first block of this slice
  int vec;                // 1: 16-byte vector path is legal
  int trans;              // 1: X = D^T (rows > cols)
};

struct PrepParams {
  PrepSlice s[kMaxSlices];
  int n_slices;
  int total_blocks;
  int step_mode;          // 1: momentum step, 0: NS-only input
  float mu;
  int nesterov;
  float eps;
  unsigned* status;
};

// ---- K6: update / copy-back --------------------------------------------------
constexpr int kFinRows = 8, kFinCols = 256;     // tile when O is stored [r][c]
constexpr int kFinTRows = 32, kFinTCols = 64;   // tile when O is read transposed from Xt
// Rows of one update tile: those of one row pass times the launch's passes
// (FinParams::passes).
constexpr int fin_tile_rows(int o_trans, int passes) { return (o_trans ? kFinTRows : kFinRows) * passes; }

struct FinSlice {
  void* W;                     // step: weights [count][r][c]; ns: output
  const __nv_bfloat16* O;      // NS result (workspace Xt): [r][c], or [c][r] when o_trans
  const __nv_bfloat16* O_lo;   // high-precision mode: its lo half (same layout), else null
  const float* inv;            // [count] extra factor when steps == 0, else null
  int64_t r, c, pitch_o, mstride_o;
  int count;
  int w_dtype;
  int tiles_r, tiles_c, tile_base;
  int vec;
  float scale;                 // update scale s(r, c)
  int o_trans;                 // 1: O[r][c] = Xt[c][r] (stored rows <= cols)
};

struct FinParams {
  FinSlice s[kMaxSlices];
  int n_slices;
  int total_blocks;
  int step_mode;
  float lr, wd;
  unsigned* status;            // device status word (debug-build checks)
  int passes;                  // row passes per tile: 2 (every W bf16) or 1; 0 reads as 1
};

// ---- NS GEMM phases -----------------------------------------------------------
enum Epi : int { kEpiGram = 0, kEpiPoly = 1, kEpiApply = 2 };

struct alignas(128) GemmGroup {
  CUtensorMap mapA;       // operand A: K-major (rows = M dim, inner = K), box 64 x 128;
                          // gram: Xt viewed MN-major (inner = m, rows = n), box 64 x 64
  CUtensorMap mapB;       // operand B: K-major box 64 x 256; gram: as mapA
  CUtensorMap mapC;       // output, box 64 x 128 (TMA store): gram A, poly B, apply Xt_new
  CUtensorMap mapD;       // gram / poly: the output's transposed boxes, box 64 x 64
  // high-precision mode: the lo halves of mapA, mapB, mapC, mapD
  CUtensorMap mapAlo, mapBlo, mapClo, mapDlo;
  const float* inv;              // first iteration scale (per matrix) or null
  float* partial;                // gram split-K partials
  unsigned* tile_cnt;            // gram split-K arrival counters
  int m, n;
  int count;
  int tiles_per_mat;
  int tile_base;
  int nt;          // apply: tiles along m (N dim); symmetric: column tiles
  int mt;          // apply: tiles along n (M dim); symmetric: row tiles
  int ksplit, kb_per_split, num_kb;
};

struct GemmParams {
  GemmGroup g[kMaxNsGroups];
  int n_groups;
  int total_tiles;
  float a, b, c;           // apply uses a - alpha; poly adds alpha on the diagonal
  float alpha;             // shift: X' = (a - alpha) X + (b A + c A^2 + alpha I) X
  int first;              // 1: operands are unnormalised, apply inv scale
  int deep;               // 1: 4-stage ring, one staging box per epilogue set
  int prec;               // 1: hi + lo operands, three K segments per product
  int inject;             // testing hook: CTA 0 arms its first ring stage and issues no
                          // copy for it, so the wait on it runs out (then the status bit)
  int pair;               // 1: clusters of two CTAs share the B tile (tiles count pair
                          // tiles; mapB holds 128-row boxes for K-major B; no split-K)
  int wide;               // 1: one CTA per 256 x 256 block, both 128-row halves (tiles count
                          // pair tiles; maps as for single tiles; bf16, no split-K)
  int b_mn;               // 1 (polynomial / apply): B is read MN-major from 64 x 64 boxes,
                          // so the product is A B rather than A B^T (B not symmetric)
  unsigned* status;
  unsigned long long timeout_ns;
};

// One core-shape group of the GEMM path on the device: workspace buffers,
// split-K plan and tensor maps (ns_plan.cpp).
struct NsGroupDev {
  int64_t m = 0, n = 0, cnt = 0, m_pad = 0;
  __nv_bfloat16* Xt[2] = {nullptr, nullptr};   // [cnt][n][m_pad] ping-pong
  __nv_bfloat16* A = nullptr;                  // [cnt][m][m_pad]
  __nv_bfloat16* B = nullptr;                  // [cnt][m][m_pad]
  const float* inv = nullptr;                  // [cnt] 1 / (||X0|| + eps)
  float* partial = nullptr;                    // Gram split-K partials
  unsigned* tile_cnt = nullptr;                // Gram split-K counters
  int ksplit = 1, kb_per_split = 1, num_kb_gram = 1;
  int64_t tri = 1;
  CUtensorMap map_gram[2], map_xt[2], map_ap, map_aq, map_a64, map_bp, map_bq, map_b64;
  // high-precision mode: lo halves of Xt, A and B (null otherwise) and their maps
  __nv_bfloat16* Xt_lo[2] = {nullptr, nullptr};
  __nv_bfloat16* A_lo = nullptr;
  __nv_bfloat16* B_lo = nullptr;
  CUtensorMap lo_gram[2], lo_xt[2], lo_ap, lo_aq, lo_a64, lo_bp, lo_bq, lo_b64;
  // Gram-space NS (gram_space = 1): five m x m bf16 matrices per problem,
  // [cnt][m][m_pad] each -- R (the Gram matrix), T = R B', B' (shifted step
  // polynomial) and Q ping-pong -- with 128-, 256- and 64-row boxes.
  int gram_space = 0;
  __nv_bfloat16* S[5] = {nullptr, nullptr, nullptr, nullptr, nullptr};
  CUtensorMap s_p[5], s_64[5];
};

// Gram-space buffers of NsGroupDev::S.
constexpr int kGsR = 0, kGsT = 1, kGsB = 2, kGsQ0 = 3;   // Q ping-pong: kGsQ0, kGsQ0 + 1

// Tiled bf16/f32 tensor map of a [dims[2]][dims[1]][dims[0]] tensor with
// byte strides strides[0] (rows) and strides[1] (matrices).
bool encode_tiled(CUtensorMap* map, bool f32, const void* base, const uint64_t* dims,
                  const uint64_t* strides, const uint32_t* box, bool swizzle128);
// bf16, 128-byte swizzle, box {64, box_rows, 1}.
bool make_ns_map(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t cnt,
                 int64_t pitch, int64_t mstride, int box_rows);
bool ns_group_maps(NsGroupDev& g);
// Fill the launch descriptor of group g for `phase` (Epi) of NS step `it`.
// pair: the launch runs in CTA pairs (see GemmParams::pair).
// wide: tiles count pair tiles (GemmParams::wide), maps as for single tiles.
void ns_fill_group(GemmGroup& G, const NsGroupDev& g, int phase, int it, int tile_base,
                   bool pair = false, bool wide = false);
// Gram-space NS (the m x m products on the polynomial kernel):
//   the Gram R = X X^T of the iterate in Xt[src] into S[kGsR];
bool ns_gs_maps(NsGroupDev& g);
void ns_fill_gs_gram(GemmGroup& G, const NsGroupDev& g, int src, int tile_base, bool pair,
                     bool wide = false);
//   C = epilogue(S[a] S[b]) into S[c] (B read MN-major, GemmParams::b_mn), with
//   the polynomial kernel's epilogue b' S[a] + c' (S[a] S[b]) + alpha' I;
void ns_fill_gs_sym(GemmGroup& G, const NsGroupDev& g, int a, int b, int c, int tile_base,
                    bool pair, bool wide = false);
//   the apply Xt[src] S[q] (the iterate times Q) into Xt[src ^ 1].
void ns_fill_gs_apply(GemmGroup& G, const NsGroupDev& g, int q, int src, int tile_base,
                      bool pair, bool wide = false);

// ---- fused small-m path: Gram-space Newton-Schulz -------------------------------
constexpr int kSmallMaxM = 64;             // core shapes with m <= 64
constexpr int kSmallThreads = 320;         // warp 0 loads, 1 MMA, 2..9 consumers
constexpr int kSmallCons = 256;            // consumer threads (a multiple of 128)
constexpr int kSmallTmemCols = 512;        // Gram accumulators [0,128); O slot s at 128 + s * tcol
constexpr int kSmallMaxStages = 8;
constexpr int kSmallCtrSlots = 64;         // ring of per-launch counter slots
constexpr int kSmallMaxSlices = 16;        // slices per launch (their tensor maps are parameters)
constexpr int kSmallSmemLimit = 227 * 1024;

struct SmallSlice {
  const void* G;     // step: gradient; NS only: the input
  float* Mom;        // step mode only
  void* W;           // step: weights; NS only: the output
  int count;         // matrices in this slice
  int mat_base;      // index of its first matrix within the launch
  int trans;         // stored rows > cols
  int g_dtype, w_dtype;
  int gbulk;         // G and Mom tiles move by TMA (tensor maps tm[.][0], tm[.][1])
  int wbulk;         // W tiles move by TMA (tensor map tm[.][2])
  float scale;       // update scale s(rows, cols)
};

struct SmallParams {
  // per slice: tiles of G and Mom (box: cw1 X columns x m rows) and of W (box:
  // 128 X columns x m rows), in the stored layout
  alignas(128) CUtensorMap tm[kSmallMaxSlices][3];
  SmallSlice s[kSmallMaxSlices];
  int n_slices;
  int m, n;          // core shape, m <= n
  int mr;            // X rows held: m rounded up to 8
  int mp;            // leading dimension of the Gram-space fp32 matrices: 32 (m <= 32) or 64
  int nmm;           // MMA N (and apply K): m rounded up to 16
  int wb;            // X columns per work item (multiple of 128)
  int nb;            // work items per matrix
  int cw1;           // X columns per first-phase stage (128, or 64 when m > 32)
  int stages;        // ring stages
  int total_mats;
  int items;         // total_mats * nb
  int xbytes;        // one item's X0 image: (wb / 64) * mr * 128
  int x_off;         // X0 tile inside a stage (1024-aligned); a zero gap follows it
  int qbytes;        // one Q image: hi and lo, nmm rows x 128 bytes each
  int pstride;       // floats per item's partial Gram blocks (2 m^2 rounded up to 4)
  int precise;       // 1: X0 kept as bf16 hi + lo (each 64-column chunk is [hi][lo])
  int nblk;          // partial Gram blocks per item (1 or 2)
  int gcols;         // TMEM columns per Gram accumulator (64, or 128 for precise m > 32);
                     // the O slots start at column 2 gcols
  int gs_lowmem;     // Gram-space job in three LD x LD buffers instead of five
  int p2_tiles;      // second phase: 128-column tiles per claim unit (a part of an item)
  int p2_units;      // second phase: most units per claim
  int p2_tma_store;  // second phase: row-major TMA-legal W' written back by TMA from the stage
  int steps;
  float coef[kMaxSteps][3];
  int step_mode, nesterov;
  float mu, lr, wd, eps;
  uint8_t* ximg;                // [items][xbytes] bf16 X0 images (shared-memory layout)
  float* part;                  // [items][pstride] partial Grams (two stacked blocks when cw1 = 128)
  uint8_t* qimg;                // [total_mats][qbytes] Q = hi + lo operand images
  unsigned* arrive;             // [2][cap]: items arrived per matrix, slot epoch % 2
  unsigned long long* ready_list;   // [total_mats] (epoch << 32) | matrix, in publication order
  unsigned* ctr;                // [kSmallCtrSlots][4]: per launch (slot epoch % slots)
                                // ready-list length, claimed second- and first-phase items
  unsigned epoch;               // this launch's tag, never 0
  int inject;                   // testing hook: the last matrix is never published, so
                                // the waits for it run out (then the status bit)
  unsigned* status;
  unsigned long long timeout_ns;
  int cap;                      // matrices per arrive slot
  // shared-memory carve-up (bytes from the 1024-aligned base)
  int off_q, off_ring, stage_bytes, off_gs, off_epi, off_bar;   // off_epi: 512 B per consumer warp
  int smem_bytes;
};

// ---- AdamW for the non-matrix parameters ------------------------------------------
struct AdamwSlice {
  void* p;                 // parameter (f32 or bf16), updated in place
  const void* g;           // gradient (f32 or bf16)
  float* m;                // first moment (fp32), updated in place
  float* v;                // second moment (fp32), updated in place
  int64_t numel;
  int64_t unit_base;       // first 8-element unit of this tensor in the launch
  int p_dtype, g_dtype;    // 0 f32, 1 bf16
  int vec;                 // 1: all four pointers 16-byte aligned
};

struct AdamwParams {
  AdamwSlice s[kMaxSlices];
  int n_slices;
  int64_t total_units;
  float lr, beta1, beta2, eps, wd;
  float step_size;         // lr / (1 - beta1^t)
  float inv_sqrt_bc2;      // 1 / sqrt(1 - beta2^t)
};

// ---- guard-band check (guard mode, a debugging aid) ------------------------------
constexpr int kGuardMaxBands = 128;
struct GuardParams {
  const uint8_t* base;             // workspace
  uint64_t off[kGuardMaxBands];    // band offsets
  int n;                           // bands
  unsigned bytes;                  // bytes per band (a multiple of 16)
  unsigned pattern;                // the byte every band holds
  unsigned long long* bad;         // += bytes found different
};

// ---- launchers (return cudaGetLastError()) ----------------------------------
cudaError_t launch_prep(const PrepParams& p, cudaStream_t s);
cudaError_t launch_finish(const FinParams& p, cudaStream_t s);
cudaError_t launch_gemm(int epi, const GemmParams& p, cudaStream_t s);
cudaError_t launch_adamw(const AdamwParams& p, int sms, cudaStream_t s);
cudaError_t launch_guard_check(const GuardParams& p, cudaStream_t s);
int gemm_block_n();      // N tile of the NS GEMMs
int gemm_block_m();      // M tile (TMEM lanes)
int gemm_block_k();      // K per pipeline stage
int gemm_sym_tiles(int m);   // tiles of a symmetric m x m product (holding some col >= row)
int gemm_sym_pair_tiles(int m);   // the same tiles taken in pairs of row tiles
// Whether a launch with `tiles` (unpaired) tiles, whose smallest core-shape
// side is min_m, runs in CTA pairs (MUON_GEMM_PAIR=0 / 1 overrides).
bool gemm_use_pair(int64_t tiles, int sms, int64_t min_m);
// Whether a bf16, unsplit grouped-GEMM launch of product `epi` runs WIDE:
// tiles = single-tile count, min_kb / mean_kb = the least and the
// tile-weighted mean number of 64-wide K blocks per tile (ns_plan.cpp).
bool gemm_use_wide(int epi, int64_t tiles, int sms, int min_kb, double mean_kb);
// Ring depth of a launch (GemmParams::deep): the Gram and the apply always
// take the 4-stage ring (their epilogues need one staging box per set); the
// polynomial, whose mirrored output wants two boxes per set in flight, only
// when every tile has at least 32 K blocks (measured on the MoE-expert and
// Llama-shaped workloads).
inline int gemm_deep(int phase, int min_kblocks) {
  return (phase != kEpiPoly || min_kblocks >= 32) ? 1 : 0;
}
cudaError_t launch_small(const SmallParams& p, int grid, cudaStream_t s);

// ---- failure-path testing hook (muon_debug_inject_stall) -------------------------
constexpr int kInjectGemm = 1;    // the next grouped-GEMM launch stalls one ring stage
constexpr int kInjectSmall = 2;   // the next small-m launch withholds one matrix
// 1 (and the request is cleared) when a stall of `kind` was requested, else 0.
int take_injected_stall(int kind);

// Device address of the allocation-free entry point's status word on device
// `dev`, or null before that entry point's first call there (noalloc.cu).
unsigned* noalloc_status_word(int dev);
int small_blocks_per_sm(int smem_bytes, bool precise);   // resident CTAs per SM, 0 on failure

}  // namespace muon
