// Tensor-core GEMMs of one Newton-Schulz step (HyperParallel-FSDP section 2.3,
// Eq. (1), evaluated as A = X X^T; B' = b*A + c*A^2 + alpha*I;
// X' = (a - alpha)*X + B' X).  The iterate is kept in one layout only,
// Xt = X^T ([n][m], m <= n), ping-ponged between two buffers:
//
//   Gram   A  = X X^T = Xt^T Xt   both operands MN-major views of Xt tiles;
//                            symmetric: only tiles holding an element with
//                            col >= row are computed, each such element is
//                            written at (r, c) and mirrored to (c, r)
//                            (DMuon-2 section 5, symmetric products);
//                            split-K over the long side for few tiles.
//   Poly   B' = b*A + c*A A + alpha*I   A is symmetric, so A A = A A^T:
//                            K-major operands; the rest is fused in the
//                            epilogue; symmetric output.  The Gram-space
//                            products (GemmParams::b_mn) read B MN-major
//                            and form S[a] S[b], not S[a] S[b]^T.
//   Apply  Xt' = (a - alpha)*Xt + Xt B'   (B' symmetric), K-major operands;
//                            the epilogue reads the Xt tile and writes the
//                            Xt' tile through shared memory with TMA.
//
// Per CTA (one per SM):
//   warp 0      TMA producer: 128x64 (P) and 256x64 (Q) tiles, 128-byte
//               swizzle, into a shared-memory ring;
//   warp 1      allocates TMEM and issues tcgen05.mma (M=128, N=256, K=16)
//               from one elected thread into one of two TMEM accumulators;
//   warps 2..9  epilogue, two sets of four warps (each set covers the 128
//               TMEM lanes and one half of the accumulator's columns):
//               tcgen05.ld, fused arithmetic.  Apply: each set stages its
//               half tile in shared memory (TMA load of Xt, in-place update,
//               TMA store of Xt').  Gram / Poly: 16-byte stores of the
//               upper part and a per-warp shared-memory transpose for the
//               mirrored copy; the polynomial's A operand is loaded before
//               the accumulator is waited for.
// The two accumulators let the epilogue of tile t overlap the mainloop of
// tile t+1.  Long-K launches run in WIDE blocks instead: both 128-row halves
// of a 256 x 256 block from one stage, one accumulator per half (see the
// kernel's template parameters).  Tiles of all matrices of all core-shape
// groups of a chunk form one static round-robin schedule, ordered in column
// groups (decode) so that the CTAs running at one time share operand panels
// in L2.  Every wait is bounded; on a timeout a status bit is set, in-flight
// copies are drained, TMEM is freed and the CTA returns.
#include "muon_internal.h"
#include "sm100_ptx.cuh"

namespace muon {

namespace {

constexpr int BM = 128;          // MMA M = TMEM lanes
constexpr int BN = 256;          // MMA N = TMEM columns per accumulator
constexpr int BK = 64;           // one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;       // K per tcgen05.mma (kind::f16)
constexpr int kABytes = BM * BK * 2;
constexpr int kBBytes = BN * BK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kEpiWarp0 = 2;
constexpr int kEpiWarps = 8;                 // two sets of four
constexpr int kEpiThreads = kEpiWarps * 32;
constexpr int kThreads = (kEpiWarp0 + kEpiWarps) * 32;
constexpr int kSetCols = BN / 2;             // accumulator columns per epilogue set
constexpr int kChunkBytes = 64 * 128;      // 64 rows of 128 bytes (one MN-major operand chunk)
constexpr int kBoxBytes = BM * 128;        // apply staging: 128 rows x 64 columns of bf16

// Shared-memory carve-up: the operand ring and the epilogue's output staging.
// Short-K launches take a 3-stage ring and 32 KB of staging per epilogue set
// (two boxes: both halves of the set's columns, or a tile half and its
// transpose, in flight together); long-K launches (DEEP) take a 4-stage ring
// and one 16 KB box per set, which the set's stores then use in turn.
//
// WIDE launches (one CTA per 256 x 256 block, both 128-row halves) take a
// 3-stage ring of 64 KB stages (two A tiles and the B tile) and one box per
// set.
template <bool DEEP, bool WIDE = false>
struct Layout {
  static constexpr int a_bytes = WIDE ? 2 * kABytes : kABytes;   // A tiles per stage
  static constexpr int stage_bytes = a_bytes + kBBytes;
  static constexpr int stages = WIDE ? 3 : (DEEP ? 4 : 3);
  static constexpr int set_bytes = (DEEP || WIDE) ? kBoxBytes : 2 * kBoxBytes;
  static constexpr int bar_off = stages * stage_bytes + 2 * set_bytes;
  static constexpr int smem = bar_off + 256 + 1024;
};
constexpr uint32_t kTmemCols = 2 * BN;
constexpr int kApplyGroup = 16;   // apply: row tiles per group of the tile order
constexpr int kSymGroup = 8;      // Gram / polynomial: column blocks per group

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, unsigned* status,
                                             unsigned long long timeout_ns, bool honour_abort) {
  const uint32_t addr = ptx::smem_u32(bar);
  if (ptx::mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(addr, parity)) return true;
    if ((it & 255u) == 0) {
      if (honour_abort && *abort_flag) return false;
      if (ptx::globaltimer() - t0 > timeout_ns) {
        atomicOr(status, kDevTimeout);
        *abort_flag = 1;
        return false;
      }
    }
  }
}

__device__ __forceinline__ void epi_bar() {   // the epilogue warps only
  asm volatile("bar.sync 1, %0;" ::"n"(kEpiThreads) : "memory");
}

struct TileInfo {
  int gi, mat, row_tile, col_tile, ksp, sym_idx, kb0, nkb;
};

// Symmetric products: column block j (BN wide) needs row blocks
// i < min(ntr, (BN*j + BN - 1)/BM + 1), i.e. the tiles holding some col >= row.
__device__ __forceinline__ int sym_rows(int j, int ntr) {
  const int r = (BN * j + BN - 1) / BM + 1;
  return r < ntr ? r : ntr;
}

// Debug builds: the decoded tile lies in its group -- matrix index, row tile
// (a pair's second row tile may be one past the last), column tile, split and
// K-block range.  Every TMA coordinate derives from these as a multiple of 64
// elements, which keeps its innermost coordinate 16-byte aligned.
template <int EPI, bool PAIR>
__device__ __forceinline__ bool tile_in_range(const GemmParams& p, const TileInfo& t) {
  if (t.gi < 0 || t.gi >= p.n_groups) return false;
  const GemmGroup& G = p.g[t.gi];
  return t.mat >= 0 && t.mat < G.count && t.row_tile >= 0 && t.row_tile < G.mt + (PAIR ? 1 : 0) &&
         t.col_tile >= 0 && t.col_tile < G.nt && t.kb0 >= 0 && t.nkb >= 0 &&
         t.kb0 + t.nkb <= G.num_kb && (EPI != kEpiGram || (t.ksp >= 0 && t.ksp < G.ksplit));
}

// PAIR: `tile` numbers pair tiles (two row tiles sharing a column tile, one
// per CTA of the pair); crank picks this CTA's row tile.
template <int EPI, bool PAIR>
__device__ __forceinline__ TileInfo decode(const GemmParams& p, int tile, int crank) {
  TileInfo t;
  int gi = 0;
  while (gi + 1 < p.n_groups && tile >= p.g[gi + 1].tile_base) ++gi;
  const GemmGroup& G = p.g[gi];
  t.gi = gi;
  const int local = tile - G.tile_base;
  t.mat = local / G.tiles_per_mat;
  const int r = local - t.mat * G.tiles_per_mat;
  t.ksp = 0;
  t.sym_idx = 0;
  if (EPI == kEpiApply) {
    // Rows in groups of kApplyGroup row units (row tiles, or pair rows),
    // column-major inside a group: the ~152 tiles in flight at a time share
    // ~16 A panels and ~10 B panels (128 x K and 256 x K bf16 each), which
    // stay in L2 even at K = 16384, instead of streaming every B panel once
    // per row tile.
    const int units = PAIR ? (G.mt + 1) / 2 : G.mt;
    constexpr int kGR = PAIR ? kApplyGroup / 2 : kApplyGroup;
    const int span = kGR * G.nt;
    const int g = r / span;
    const int local = r - g * span;
    const int ge = min(kGR, units - g * kGR);
    t.col_tile = local / ge;
    const int ru = g * kGR + (local - t.col_tile * ge);
    t.row_tile = PAIR ? 2 * ru + crank : ru;
  } else {
    int idx = r / G.ksplit;
    t.ksp = r - idx * G.ksplit;
    t.sym_idx = idx;
    // Column blocks in groups of kSymGroup; inside a group, row units (row
    // tiles, or pair rows) outer and the group's columns inner, each tile
    // holding some col >= row once: unit u lies in column j iff u < rows(j),
    // rows(j) = min(units, 2j + 2) (pair rows: min(units, j + 1)), i.e. iff
    // j >= jmin(u) = u / 2 (pair rows: u).  The tiles in flight share a few
    // A and B panels, as in the apply's order.
    const int units = PAIR ? (G.mt + 1) / 2 : G.mt;
    auto rows_u = [&](int j) { return min(units, PAIR ? j + 1 : 2 * j + 2); };
    auto jmin = [&](int u) { return PAIR ? u : u >> 1; };
    const int ntc = G.nt;
    int j0 = 0, j1 = 0, w = 0, full = 0;
    for (;;) {
      j1 = min(ntc, j0 + kSymGroup);
      w = j1 - j0;
      full = rows_u(j0);                 // units that hold all w columns
      int cnt = full * w;
      const int top = rows_u(j1 - 1);
      for (int u = full; u < top; ++u) cnt += j1 - jmin(u);
      if (idx < cnt || j1 >= ntc) break;
      idx -= cnt;
      j0 = j1;
    }
    int u, j;
    if (idx < full * w) {
      u = idx / w;
      j = j0 + (idx - u * w);
    } else {
      idx -= full * w;
      for (u = full;; ++u) {
        const int c = j1 - jmin(u);
        if (idx < c) break;
        idx -= c;
      }
      j = jmin(u) + idx;
    }
    t.row_tile = PAIR ? 2 * u + crank : u;
    t.col_tile = j;
  }
  t.kb0 = t.ksp * G.kb_per_split;
  const int e = t.kb0 + G.kb_per_split < G.num_kb ? t.kb0 + G.kb_per_split : G.num_kb;
  t.nkb = e - t.kb0;
  return t;
}

__device__ __forceinline__ void cvt_bf16x32(const uint4 (&u)[4], float* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u[q]);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      v[8 * q + 2 * k] = f.x;
      v[8 * q + 2 * k + 1] = f.y;
    }
  }
}


}  // namespace

// PREC: the high-precision mode.  Every operand is a pair of bf16 tensors
// (hi, lo) and each product runs over three K segments, hi*hi, hi*lo and
// lo*hi, into one fp32 accumulator; the epilogue reads hi + lo and writes the
// result again as hi = bf16(v), lo = bf16(v - hi).  Shallow layout only.
//
// PAIR: CTAs run in clusters of two on two row tiles that share a column tile
// (a 256 x 256 output block).  Each CTA loads its own 128-row A tile and one
// half of the common 256-row B tile, which TMA multicasts into the same
// stage of both CTAs, so every CTA reads 32 KB instead of 48 KB per K block
// from L2.  Each CTA still issues its own M = 128 MMAs into its own TMEM; a
// stage is refilled once the MMAs of BOTH CTAs are done with it (each MMA
// issuer's commit arrives on both CTAs' empty barrier, count 2).  The pair
// passes a cluster barrier after initialising its mbarriers and before
// exiting, so no copy or arrival ever targets a CTA that is not running.
//
// WIDE: one CTA computes both 128-row halves of a 256 x 256 block (the pair
// tiles above, without a partner).  Each stage holds the two A tiles and the
// common B tile, and the MMA issuer runs both halves' MMAs on it, half h into
// accumulator h: 64 KB of operands per two 128 x 256 x 64 MMA blocks instead
// of 48 KB per one, a third less operand data into the SM per MMA.  Both
// accumulators belong to one block, so a block's MMAs start once the
// epilogue has drained both; the epilogue sees the halves as consecutive
// tiles (virtual tile 2n + h).
template <int EPI, bool DEEP, bool PREC, bool PAIR, bool WIDE = false>
__global__ void __launch_bounds__(kThreads, 1) ns_gemm_kernel(const __grid_constant__ GemmParams p) {
  static_assert(!(WIDE && (PAIR || PREC)), "WIDE runs alone, in bf16");
  constexpr bool kPT = PAIR || WIDE;   // tiles are pair tiles
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  using L = Layout<DEEP, WIDE>;
  constexpr int kStages = L::stages;
  constexpr int kAB = L::a_bytes;
  constexpr int kSB = L::stage_bytes;
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kAB;
  uint8_t* sX = smem + kStages * kSB;   // epilogue output staging
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + L::bar_off);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;      // [2] accumulator ready
  uint64_t* tempty = tfull + 2;           // [2] accumulator drained
  uint64_t* xfull = tempty + 2;           // [2] apply: staged Xt tile of epilogue set s landed
  uint64_t* mma_drain = xfull + 2;        // the MMA issuer's last MMAs have completed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(mma_drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_last = reinterpret_cast<int*>(tmem_slot + 2);
  volatile int* s_ok = reinterpret_cast<volatile int*>(tmem_slot + 3);   // [2] per-tile decision

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int crank = PAIR ? static_cast<int>(ptx::cluster_ctarank()) : 0;
  const int tile0 = PAIR ? static_cast<int>(blockIdx.x >> 1) : static_cast<int>(blockIdx.x);
  const int tstep = PAIR ? static_cast<int>(gridDim.x >> 1) : static_cast<int>(gridDim.x);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], PAIR ? 2 : 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&tfull[b], 1);
      ptx::mbar_init(&tempty[b], kEpiThreads);
      ptx::mbar_init(&xfull[b], 1);
    }
    ptx::mbar_init(mma_drain, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    for (int g = 0; g < p.n_groups; ++g) {
      ptx::prefetch_tmap(&p.g[g].mapA);
      ptx::prefetch_tmap(&p.g[g].mapB);
      ptx::prefetch_tmap(&p.g[g].mapC);
      if (EPI != kEpiApply) ptx::prefetch_tmap(&p.g[g].mapD);
      if (PREC) {
        ptx::prefetch_tmap(&p.g[g].mapAlo);
        ptx::prefetch_tmap(&p.g[g].mapBlo);
        ptx::prefetch_tmap(&p.g[g].mapClo);
        if (EPI != kEpiApply) ptx::prefetch_tmap(&p.g[g].mapDlo);
      }
    }
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  if (PAIR) ptx::cluster_sync();   // both CTAs' mbarriers are initialised
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- TMA producer ------------------------------------------------------------------
    if (lane == 0) {
      constexpr int NSEG = PREC ? 3 : 1;   // K segments: (hi, hi), (hi, lo), (lo, hi)
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool stop = false;
      for (int tile = tile0; tile < p.total_tiles && !stop; tile += tstep) {
        const TileInfo t = decode<EPI, kPT>(p, tile, crank);
        if (!dbg_ok(tile_in_range<EPI, kPT>(p, t), p.status)) break;   // consumers time out
        const GemmGroup& G = p.g[t.gi];
        for (int i = 0; i < t.nkb * NSEG; ++i) {
          if (!wait_bounded(&empty[stage], phase ^ 1, abort_flag, p.status, p.timeout_ns, true)) {
            stop = true;
            break;
          }
          const int seg = PREC ? i / t.nkb : 0;
          const int kx = (t.kb0 + i - seg * t.nkb) * BK;
          const CUtensorMap* ma = (PREC && seg == 2) ? &G.mapAlo : &G.mapA;
          const CUtensorMap* mb = (PREC && seg == 1) ? &G.mapBlo : &G.mapB;
          if (p.inject && blockIdx.x == 0 && issued == 0) {
            // testing hook: this stage is never armed and no copy is issued
            // for it, so the MMA issuer's wait on it runs out
          } else if (EPI == kEpiGram) {
            ptx::mbar_arrive_expect_tx(&full[stage], kSB);
            // MN-major chunks of Xt: 64 columns (m) x 64 rows (n, the K dim)
            // each; WIDE: both 128-row halves (half h at kABytes h)
#pragma unroll
            for (int h = 0; h < (WIDE ? 2 : 1) * BM / 64; ++h)
              ptx::tma_load_3d(sA + stage * kAB + h * kChunkBytes, ma, &full[stage],
                               t.row_tile * BM + 64 * h, kx, t.mat);
            if (PAIR) {
              // this CTA's half of the B chunks, into both CTAs of the pair
#pragma unroll
              for (int h = 2 * crank; h < 2 * crank + 2; ++h)
                ptx::tma_load_3d_mc(sB + stage * kBBytes + h * kChunkBytes, mb, &full[stage],
                                    t.col_tile * BN + 64 * h, kx, t.mat, 0x3);
            } else {
#pragma unroll
              for (int h = 0; h < BN / 64; ++h)
                ptx::tma_load_3d(sB + stage * kBBytes + h * kChunkBytes, mb, &full[stage],
                                 t.col_tile * BN + 64 * h, kx, t.mat);
            }
          } else {
            ptx::mbar_arrive_expect_tx(&full[stage], kSB);
#pragma unroll
            for (int hh = 0; hh < (WIDE ? 2 : 1); ++hh)   // WIDE: both 128-row halves
              ptx::tma_load_3d(sA + stage * kAB + hh * kABytes, ma, &full[stage], kx,
                               (t.row_tile + hh) * BM, t.mat);
            if (p.b_mn) {
              // B[k][col] in MN-major chunks of 64 columns x 64 rows (K), as the Gram's B
              for (int h = PAIR ? 2 * crank : 0; h < (PAIR ? 2 * crank + 2 : BN / 64); ++h) {
                if (PAIR)
                  ptx::tma_load_3d_mc(sB + stage * kBBytes + h * kChunkBytes, mb, &full[stage],
                                      t.col_tile * BN + 64 * h, kx, t.mat, 0x3);
                else
                  ptx::tma_load_3d(sB + stage * kBBytes + h * kChunkBytes, mb, &full[stage],
                                   t.col_tile * BN + 64 * h, kx, t.mat);
              }
            } else if (PAIR)   // B rows [BN/2 crank, BN/2 crank + BN/2) of the tile (128-row box)
              ptx::tma_load_3d_mc(sB + stage * kBBytes + crank * (kBBytes / 2), mb, &full[stage], kx,
                                  t.col_tile * BN + crank * (BN / 2), t.mat, 0x3);
            else
              ptx::tma_load_3d(sB + stage * kBBytes, mb, &full[stage], kx, t.col_tile * BN, t.mat);
          }
          ++issued;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
      }
      // drain: the last (up to) kStages issued copies have landed before exit
      for (int j = issued > kStages ? issued - kStages : 0; j < issued; ++j)
        wait_bounded(&full[j % kStages], (j / kStages) & 1, abort_flag, p.status, p.timeout_ns,
                     false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer --------------------------------------------------------------------
    if (lane == 0) {
      // the Gram reads both operands MN-major (A and B transpose bits)
      const bool b_mn = EPI == kEpiGram || p.b_mn;
      const uint32_t idesc = ptx::idesc_bf16_f32(BM, BN) | (EPI == kEpiGram ? 1u << 15 : 0u) |
                             (b_mn ? 1u << 16 : 0u);
      int stage = 0, acc = 0;
      uint32_t phase = 0;
      bool stop = false;
      // WIDE: a block takes both accumulators (virtual tiles acc, acc + 1)
      for (int tile = tile0; tile < p.total_tiles && !stop; tile += tstep, acc += WIDE ? 2 : 1) {
        const TileInfo t = decode<EPI, kPT>(p, tile, crank);
        const int buf = acc & 1;
        if (!wait_bounded(&tempty[buf], ((acc >> 1) & 1) ^ 1, abort_flag, p.status, p.timeout_ns,
                          true) ||
            (WIDE && !wait_bounded(&tempty[1], ((acc >> 1) & 1) ^ 1, abort_flag, p.status,
                                   p.timeout_ns, true))) {
          stop = true;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + buf * BN;
        for (int i = 0; i < t.nkb * (PREC ? 3 : 1); ++i) {
          if (!wait_bounded(&full[stage], phase, abort_flag, p.status, p.timeout_ns, true)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(sA + stage * kAB);
          const uint32_t b0 = ptx::smem_u32(sB + stage * kBBytes);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k) {
            // K-major: K advances within the 128-byte row; MN-major: by 16
            // rows (two 1024-byte swizzle atoms) within each 64-column chunk
            const uint64_t da = EPI == kEpiGram
                                    ? ptx::sdesc_mnmajor_sw128(a0 + k * 2048, kChunkBytes, 1024)
                                    : ptx::sdesc_kmajor_sw128(a0 + k * UMMA_K * 2);
            const uint64_t db = b_mn
                                    ? ptx::sdesc_mnmajor_sw128(b0 + k * 2048, kChunkBytes, 1024)
                                    : ptx::sdesc_kmajor_sw128(b0 + k * UMMA_K * 2);
            ptx::umma_bf16(d, da, db, idesc, (i > 0 || k > 0) ? 1u : 0u);
            if (WIDE) {   // the second half's A tile, same B, into accumulator 1
              const uint64_t da1 =
                  EPI == kEpiGram
                      ? ptx::sdesc_mnmajor_sw128(a0 + kABytes + k * 2048, kChunkBytes, 1024)
                      : ptx::sdesc_kmajor_sw128(a0 + kABytes + k * UMMA_K * 2);
              ptx::umma_bf16(tmem + BN, da1, db, idesc, (i > 0 || k > 0) ? 1u : 0u);
            }
          }
          if (PAIR) ptx::umma_commit_mc(&empty[stage], 0x3);   // both CTAs' stage
          else ptx::umma_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        ptx::umma_commit(&tfull[buf]);   // accumulator complete (or abandoned)
        if (WIDE) ptx::umma_commit(&tfull[1]);
      }
      // no MMA may still run when TMEM is freed (after an abort nobody
      // waits for the last accumulator)
      ptx::umma_commit(mma_drain);
      wait_bounded(mma_drain, 0, abort_flag, p.status, p.timeout_ns, false);
    }
    __syncwarp();
  } else {
    // ---- epilogue (warps 2..9; TMEM lane quadrant = warp % 4, column half = set) ----------
    const int q4 = warp & 3;
    const int set = (warp - kEpiWarp0) >> 2;
    const int cbase = set * kSetCols;
    const int row = q4 * 32 + lane;
    const bool leader = (warp - kEpiWarp0) % 4 == 0 && lane == 0;   // one thread per set
    uint8_t* stg = sX + set * L::set_bytes;    // this set's staging
    uint32_t xphase = 0;
    bool xpend = false;   // leader: a staged-tile load is in flight and not yet waited for
    int acc = 0;
    // WIDE: virtual tile vt is half vt & 1 of block vt >> 1 (accumulator vt & 1)
    for (int vt = 0;; ++vt, ++acc) {
      const int tile = tile0 + (WIDE ? (vt >> 1) : vt) * tstep;
      if (tile >= p.total_tiles) break;
      const TileInfo t = decode<EPI, kPT>(p, tile, WIDE ? (vt & 1) : crank);
      const GemmGroup& G = p.g[t.gi];
      const int buf = acc & 1;
      const int row0 = t.row_tile * BM, col0 = t.col_tile * BN;
      // Apply: the Xt tile half of this set does not depend on the
      // accumulator, so the leader requests it first (once the previous
      // tile's stores have read the staging boxes).
      if (EPI == kEpiApply && leader && !xpend && !*abort_flag) {
        xpend = true;
        ptx::bulk_wait_read<0>();
        if (PREC) {
          // the first half's hi and lo boxes
          ptx::mbar_arrive_expect_tx(&xfull[set], 2 * kBoxBytes);
          ptx::tma_load_3d(stg, &G.mapA, &xfull[set], col0 + cbase, row0, t.mat);
          ptx::tma_load_3d(stg + kBoxBytes, &G.mapAlo, &xfull[set], col0 + cbase, row0, t.mat);
        } else {
          constexpr int nh = DEEP ? 1 : 2;    // halves staged now
          ptx::mbar_arrive_expect_tx(&xfull[set], nh * kBoxBytes);
#pragma unroll
          for (int h = 0; h < nh; ++h)
            ptx::tma_load_3d(stg + h * kBoxBytes, &G.mapA, &xfull[set], col0 + cbase + 64 * h,
                             row0, t.mat);
        }
      }
      wait_bounded(&tfull[buf], (acc >> 1) & 1, abort_flag, p.status, p.timeout_ns, false);
      // One decision for all epilogue warps (they share named barriers): one
      // thread samples the abort flag, the barrier publishes it.  The slot
      // alternates, so it is rewritten only after everyone passed the next
      // tile's barrier (and so had read it).
      if (threadIdx.x == kEpiWarp0 * 32) s_ok[acc & 1] = !*abort_flag;
      epi_bar();
      const bool ok = s_ok[acc & 1] != 0;
      ptx::tc_fence_after();
      const uint32_t taddr = tmem + buf * BN + (static_cast<uint32_t>(q4 * 32) << 16);
      if (!ok) {
        ptx::tc_fence_before();
        ptx::mbar_arrive(&tempty[buf]);
        break;
      }
      if (EPI == kEpiApply && PREC) {
        const float s = p.first ? G.inv[t.mat] : 1.f;
        for (int h = 0; h < 2; ++h) {
          // box 0: hi, box 1: lo of this half (64 columns)
          if (h == 1 && leader && !xpend && !*abort_flag) {
            xpend = true;
            ptx::bulk_wait_read<0>();
            ptx::mbar_arrive_expect_tx(&xfull[set], 2 * kBoxBytes);
            ptx::tma_load_3d(stg, &G.mapA, &xfull[set], col0 + cbase + 64, row0, t.mat);
            ptx::tma_load_3d(stg + kBoxBytes, &G.mapAlo, &xfull[set], col0 + cbase + 64, row0, t.mat);
          }
          const bool xok = wait_bounded(&xfull[set], xphase, abort_flag, p.status, p.timeout_ns, false);
          if (xok) {
            xphase ^= 1u;
            xpend = false;
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int c0 = cbase + 64 * h + 32 * cc;
              uint32_t r[32];
              ptx::tmem_ld_32x32b_x32(taddr + c0, r);
              ptx::tmem_ld_wait();
              uint32_t off[4];
              uint4 xh[4], xl[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                off[q] = ptx::sw128_offset(row, (cc * 4 + q) * 16);
                xh[q] = *reinterpret_cast<const uint4*>(stg + off[q]);
                xl[q] = *reinterpret_cast<const uint4*>(stg + kBoxBytes + off[q]);
              }
              float x[32], xlo[32];
              cvt_bf16x32(xh, x);
              cvt_bf16x32(xl, xlo);
              __align__(16) __nv_bfloat16 hv[32], lv[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const float v = s * fmaf(p.a, x[j] + xlo[j], __uint_as_float(r[j]));
                hv[j] = __float2bfloat16_rn(v);
                lv[j] = __float2bfloat16_rn(v - __bfloat162float(hv[j]));
              }
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                *reinterpret_cast<uint4*>(stg + off[q]) = *reinterpret_cast<const uint4*>(hv + 8 * q);
                *reinterpret_cast<uint4*>(stg + kBoxBytes + off[q]) =
                    *reinterpret_cast<const uint4*>(lv + 8 * q);
              }
            }
          }
          if (h == 1) {
            ptx::tc_fence_before();
            ptx::mbar_arrive(&tempty[buf]);
          }
          ptx::fence_proxy_async_smem();
          ptx::named_bar(2 + set, 128);
          if (leader && xok) {
            const int x = col0 + cbase + 64 * h;
            if (x < G.m && row0 < G.n) {
              ptx::tma_store_3d(&G.mapC, stg, x, row0, t.mat);
              ptx::tma_store_3d(&G.mapClo, stg + kBoxBytes, x, row0, t.mat);
            }
            ptx::bulk_commit();
          }
        }
      } else if (EPI == kEpiApply) {
        const float s = p.first ? G.inv[t.mat] : 1.f;
        for (int h = 0; h < 2; ++h) {
          uint8_t* box = stg + (DEEP ? 0 : h * kBoxBytes);
          if (DEEP && h == 1 && leader && !xpend && !*abort_flag) {
            // the first half's store has read the box: stage the second half
            xpend = true;
            ptx::bulk_wait_read<0>();
            ptx::mbar_arrive_expect_tx(&xfull[set], kBoxBytes);
            ptx::tma_load_3d(box, &G.mapA, &xfull[set], col0 + cbase + 64, row0, t.mat);
          }
          bool xok = true;
          if (!DEEP && h == 1) {
            // both halves arrived with the first wait
          } else {
            // every thread of the set waits for the staged half (bounded)
            xok = wait_bounded(&xfull[set], xphase, abort_flag, p.status, p.timeout_ns, false);
            if (xok) {
              xphase ^= 1u;
              xpend = false;
            }
          }
          if (xok) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int c0 = cbase + 64 * h + 32 * cc;   // accumulator column
              uint32_t r[32];
              ptx::tmem_ld_32x32b_x32(taddr + c0, r);
              ptx::tmem_ld_wait();
              // this row's 64 bytes of the chunk in the swizzled box
              uint32_t off[4];
              uint4 xv[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                off[q] = ptx::sw128_offset(row, (cc * 4 + q) * 16);
                xv[q] = *reinterpret_cast<const uint4*>(box + off[q]);
              }
              float x[32];
              cvt_bf16x32(xv, x);
              __align__(16) __nv_bfloat16 hv[32];
#pragma unroll
              for (int j = 0; j < 32; ++j)
                hv[j] = __float2bfloat16_rn(s * fmaf(p.a, x[j], __uint_as_float(r[j])));
#pragma unroll
              for (int q = 0; q < 4; ++q)
                *reinterpret_cast<uint4*>(box + off[q]) = *reinterpret_cast<const uint4*>(hv + 8 * q);
            }
          }
          if (h == 1) {
            ptx::tc_fence_before();
            ptx::mbar_arrive(&tempty[buf]);
          }
          // make the generic-proxy writes visible to the TMA store, then one
          // thread stores the half if it holds part of the matrix
          ptx::fence_proxy_async_smem();
          ptx::named_bar(2 + set, 128);
          if (leader && xok) {
            const int x = col0 + cbase + 64 * h;
            if (x < G.m && row0 < G.n) ptx::tma_store_3d(&G.mapC, box, x, row0, t.mat);
            ptx::bulk_commit();
          }
        }
      } else {
        const int64_t gr = (int64_t)row0 + row;
        const int64_t slot = (int64_t)t.mat * G.tiles_per_mat / G.ksplit + t.sym_idx;
        // debug builds: a slot outside the partial buffer is stored directly instead
        const bool split =
            G.ksplit > 1 &&
            dbg_ok(slot >= 0 && slot < (int64_t)G.count * (G.tiles_per_mat / G.ksplit) &&
                       t.ksp >= 0 && t.ksp < G.ksplit,
                   p.status);
        float* part = split ? G.partial + slot * G.ksplit * (int64_t)(BM * BN) : nullptr;
        if (split) {
          // partial tile -> global (valid entries only), then the last split reduces
          for (int c0 = cbase; c0 < cbase + kSetCols; c0 += 32) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(taddr + c0, r);
            ptx::tmem_ld_wait();
            if (gr < G.m) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const int64_t gc = (int64_t)col0 + c0 + j;
                if (gc < G.m)
                  __stcg(part + (int64_t)t.ksp * (BM * BN) + (c0 + j) * BM + row,
                         __uint_as_float(r[j]));
              }
            }
          }
          ptx::tc_fence_before();
          ptx::mbar_arrive(&tempty[buf]);
          __threadfence();
          epi_bar();
          if (threadIdx.x == kEpiWarp0 * 32) {
            const unsigned prev = atomicAdd(&G.tile_cnt[slot], 1u);
            *s_last = (prev == (unsigned)(G.ksplit - 1));
          }
          epi_bar();
          const bool last = *s_last != 0;
          epi_bar();   // everyone has read s_last before it can be rewritten
          if (!last) continue;
          __threadfence();
        }
        // Output: every computed tile stores its whole box (a tile that
        // crosses the diagonal thus also writes the elements below it, which
        // no other tile writes); a tile entirely above the diagonal also
        // stores its transpose, whose region no computed tile covers.  Each
        // element of the m x m result is written exactly once.
        const float scale = (EPI == kEpiGram && p.first) ? G.inv[t.mat] * G.inv[t.mat] : 1.f;
        const bool mirror = row0 + BM <= col0;
        // direct box: 128 rows x 64 columns (PREC: hi in sd, lo in sdl); the
        // transposed boxes 2 x (64 x 64) share the direct boxes' space when
        // the set has one box (DEEP) or needs both for hi and lo (PREC)
        constexpr bool kAliasMirror = DEEP || PREC;
        uint8_t* sd = stg;
        uint8_t* sdl = stg + kBoxBytes;
        uint8_t* sm = stg + (kAliasMirror ? 0 : kBoxBytes);
        for (int h = 0; h < 2; ++h) {
          const int c_h = cbase + 64 * h;   // accumulator column of this half
          const int gc_h = col0 + c_h;
          if (gc_h >= G.m) break;           // uniform within the set
          if (leader) {
            ptx::bulk_wait_read<0>();       // the previous stores have read the boxes
            if (EPI == kEpiPoly && !xpend && !*abort_flag) {
              xpend = true;
              ptx::mbar_arrive_expect_tx(&xfull[set], (PREC ? 2 : 1) * kBoxBytes);
              ptx::tma_load_3d(sd, &G.mapA, &xfull[set], gc_h, row0, t.mat);   // A tile
              if (PREC) ptx::tma_load_3d(sdl, &G.mapAlo, &xfull[set], gc_h, row0, t.mat);
            }
          }
          ptx::named_bar(2 + set, 128);
          bool xok = true;
          if (EPI == kEpiPoly) {
            xok = wait_bounded(&xfull[set], xphase, abort_flag, p.status, p.timeout_ns, false);
            if (xok) {
              xphase ^= 1u;
              xpend = false;
            }
          }
          uint4 keep[2][4];   // this row's 64 results (bf16), for the transposed copy
          uint4 keepl[PREC ? 2 : 1][4];   // PREC: their lo parts
          if (xok) {
#pragma unroll
            for (int cc = 0; cc < 2; ++cc) {
              const int c0 = c_h + 32 * cc;
              const int64_t gc0 = (int64_t)col0 + c0;
              float v[32];
              if (split) {
                // sum the splits in order; the 32 columns of a split are loaded together
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = 0.f;
                if (gr < G.m) {
                  for (int q = 0; q < G.ksplit; ++q) {
                    const float* pq = part + (int64_t)q * (BM * BN) + c0 * BM + row;
                    float l[32];
#pragma unroll
                    for (int j = 0; j < 32; ++j) l[j] = gc0 + j < G.m ? __ldcg(pq + j * BM) : 0.f;
#pragma unroll
                    for (int j = 0; j < 32; ++j) v[j] += l[j];
                  }
                }
              } else {
                uint32_t r[32];
                ptx::tmem_ld_32x32b_x32(taddr + c0, r);
                ptx::tmem_ld_wait();
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
              }
              uint32_t off[4];
#pragma unroll
              for (int q = 0; q < 4; ++q) off[q] = ptx::sw128_offset(row, (cc * 4 + q) * 16);
              if (EPI == kEpiPoly) {
                uint4 av4[4];
#pragma unroll
                for (int q = 0; q < 4; ++q) av4[q] = *reinterpret_cast<const uint4*>(sd + off[q]);
                float av[32];
                cvt_bf16x32(av4, av);
                if (PREC) {
#pragma unroll
                  for (int q = 0; q < 4; ++q) av4[q] = *reinterpret_cast<const uint4*>(sdl + off[q]);
                  float al[32];
                  cvt_bf16x32(av4, al);
#pragma unroll
                  for (int j = 0; j < 32; ++j) av[j] += al[j];
                }
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  v[j] = fmaf(p.b, av[j], p.c * v[j]) + (gr == gc0 + j ? p.alpha : 0.f);
              } else {
#pragma unroll
                for (int j = 0; j < 32; ++j) v[j] *= scale;
              }
              __align__(16) __nv_bfloat16 hv[32];
#pragma unroll
              for (int j = 0; j < 32; ++j) hv[j] = __float2bfloat16_rn(v[j]);
#pragma unroll
              for (int q = 0; q < 4; ++q) {
                keep[cc][q] = *reinterpret_cast<const uint4*>(hv + 8 * q);
                *reinterpret_cast<uint4*>(sd + off[q]) = keep[cc][q];
              }
              if constexpr (PREC) {
                __align__(16) __nv_bfloat16 lv[32];
#pragma unroll
                for (int j = 0; j < 32; ++j) lv[j] = __float2bfloat16_rn(v[j] - __bfloat162float(hv[j]));
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                  keepl[cc][q] = *reinterpret_cast<const uint4*>(lv + 8 * q);
                  *reinterpret_cast<uint4*>(sdl + off[q]) = keepl[cc][q];
                }
              }
            }
          }
          ptx::fence_proxy_async_smem();
          ptx::named_bar(2 + set, 128);
          if (leader && xok) {
            if (row0 < G.m) {   // a pair's second row tile may lie past the matrix
              ptx::tma_store_3d(&G.mapC, sd, gc_h, row0, t.mat);
              if (PREC) ptx::tma_store_3d(&G.mapClo, sdl, gc_h, row0, t.mat);
            }
            ptx::bulk_commit();
          }
          if (mirror) {
            if (kAliasMirror) {
              // the direct stores must have read the boxes first
              if (leader) ptx::bulk_wait_read<0>();
              ptx::named_bar(2 + set, 128);
            }
            if (xok) {
              // element (row, c) goes to row c, column `row` of the transpose
              uint8_t* tbox = sm + (row >> 6) * (kBoxBytes / 2);
              const uint32_t tb = static_cast<uint32_t>(row & 63) * 2;
#pragma unroll
              for (int cc = 0; cc < 2; ++cc) {
                const __nv_bfloat16* hv = reinterpret_cast<const __nv_bfloat16*>(keep[cc]);
#pragma unroll
                for (int j = 0; j < 32; ++j)
                  *reinterpret_cast<__nv_bfloat16*>(tbox + ptx::sw128_offset(cc * 32 + j, tb)) = hv[j];
                if constexpr (PREC) {
                  const __nv_bfloat16* lv = reinterpret_cast<const __nv_bfloat16*>(keepl[cc]);
#pragma unroll
                  for (int j = 0; j < 32; ++j)
                    *reinterpret_cast<__nv_bfloat16*>(tbox + kBoxBytes + ptx::sw128_offset(cc * 32 + j, tb)) =
                        lv[j];
                }
              }
            }
            ptx::fence_proxy_async_smem();
            ptx::named_bar(2 + set, 128);
            if (leader && xok) {
#pragma unroll
              for (int b = 0; b < 2; ++b)
                if (row0 + 64 * b < G.m) {
                  ptx::tma_store_3d(&G.mapD, sm + b * (kBoxBytes / 2), row0 + 64 * b, gc_h, t.mat);
                  if (PREC)
                    ptx::tma_store_3d(&G.mapDlo, sm + kBoxBytes + b * (kBoxBytes / 2), row0 + 64 * b,
                                      gc_h, t.mat);
                }
              ptx::bulk_commit();
            }
          }
        }
        if (!split) {
          ptx::tc_fence_before();
          ptx::mbar_arrive(&tempty[buf]);
        } else if (threadIdx.x == kEpiWarp0 * 32) {
          G.tile_cnt[slot] = 0u;
        }
      }
    }
    if (leader) {
      // no copy may still target or read this CTA's shared memory at exit
      if (xpend) wait_bounded(&xfull[set], xphase, abort_flag, p.status, p.timeout_ns, false);
      ptx::bulk_wait_all();
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  // the peer's copies into this CTA and its arrivals on this CTA's barriers
  // are all done once it has drained and reached this barrier
  if (PAIR) ptx::cluster_sync();
  if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
}

int gemm_block_n() { return BN; }
int gemm_block_m() { return BM; }
int gemm_block_k() { return BK; }

int gemm_sym_pair_tiles(int m) {
  const int ntr = (m + BM - 1) / BM, ntc = (m + BN - 1) / BN;
  int t = 0;
  for (int j = 0; j < ntc; ++j) {
    const int r = (BN * j + BN - 1) / BM + 1;
    t += ((r < ntr ? r : ntr) + 1) / 2;
  }
  return t;
}

int gemm_sym_tiles(int m) {
  const int ntr = (m + BM - 1) / BM, ntc = (m + BN - 1) / BN;
  int t = 0;
  for (int j = 0; j < ntc; ++j) {
    const int r = (BN * j + BN - 1) / BM + 1;
    t += r < ntr ? r : ntr;
  }
  return t;
}

template <int EPI, bool DEEP, bool PREC>
static cudaError_t launch_one(const GemmParams& p, int grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(ns_gemm_kernel<EPI, DEEP, PREC, false>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Layout<DEEP>::smem);
  if (e != cudaSuccess) return e;
  ns_gemm_kernel<EPI, DEEP, PREC, false><<<grid, kThreads, Layout<DEEP>::smem, s>>>(p);
  return cudaGetLastError();
}

// WIDE launch: one CTA per SM over the 256 x 256 blocks (pair tiles).
template <int EPI>
static cudaError_t launch_wide(const GemmParams& p, int grid, cudaStream_t s) {
  using LW = Layout<true, true>;
  auto kern = ns_gemm_kernel<EPI, true, false, false, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, LW::smem);
  if (e != cudaSuccess) return e;
  kern<<<grid, kThreads, LW::smem, s>>>(p);
  return cudaGetLastError();
}

// Paired launch: clusters of two CTAs, as many clusters as can be resident
// at once (the occupancy API's count for this kernel), at most one per pair
// tile.
template <int EPI, bool DEEP>
static cudaError_t launch_pair(const GemmParams& p, cudaStream_t s) {
  auto kern = ns_gemm_kernel<EPI, DEEP, false, true>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Layout<DEEP>::smem);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = Layout<DEEP>::smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  static int max_clusters = 0;   // per template instance
  if (max_clusters == 0) {
    cfg.gridDim = dim3(2, 1, 1);
    int n = 0;
    e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
    if (e != cudaSuccess) return e;
    if (n <= 0) return cudaErrorInvalidConfiguration;
    max_clusters = n;
  }
  const int clusters = p.total_tiles < max_clusters ? p.total_tiles : max_clusters;
  cfg.gridDim = dim3(static_cast<unsigned>(2 * clusters), 1, 1);
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

cudaError_t launch_gemm(int epi, const GemmParams& p, cudaStream_t s) {
  if (p.total_tiles <= 0) return cudaSuccess;
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (sms <= 0) sms = 1;
  }
  const int grid = p.total_tiles < sms ? p.total_tiles : sms;
  const bool deep = p.deep != 0;
  if (p.prec) {   // the high-precision mode runs on the shallow layout, unpaired
    switch (epi) {
      case kEpiGram: return launch_one<kEpiGram, false, true>(p, grid, s);
      case kEpiPoly: return launch_one<kEpiPoly, false, true>(p, grid, s);
      case kEpiApply: return launch_one<kEpiApply, false, true>(p, grid, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if (p.wide) {
    switch (epi) {
      case kEpiGram: return launch_wide<kEpiGram>(p, grid, s);
      case kEpiPoly: return launch_wide<kEpiPoly>(p, grid, s);
      case kEpiApply: return launch_wide<kEpiApply>(p, grid, s);
      default: return cudaErrorInvalidValue;
    }
  }
  if (p.pair) {
    switch (epi) {
      case kEpiGram: return deep ? launch_pair<kEpiGram, true>(p, s) : launch_pair<kEpiGram, false>(p, s);
      case kEpiPoly: return deep ? launch_pair<kEpiPoly, true>(p, s) : launch_pair<kEpiPoly, false>(p, s);
      case kEpiApply: return deep ? launch_pair<kEpiApply, true>(p, s) : launch_pair<kEpiApply, false>(p, s);
      default: return cudaErrorInvalidValue;
    }
  }
  switch (epi) {
    case kEpiGram: return deep ? launch_one<kEpiGram, true, false>(p, grid, s)
                               : launch_one<kEpiGram, false, false>(p, grid, s);
    case kEpiPoly: return deep ? launch_one<kEpiPoly, true, false>(p, grid, s)
                               : launch_one<kEpiPoly, false, false>(p, grid, s);
    case kEpiApply: return deep ? launch_one<kEpiApply, true, false>(p, grid, s)
                                : launch_one<kEpiApply, false, false>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace muon
