// Host-side pieces of the grouped GEMM path shared by the allocating entry
// points (api.cpp) and the allocation-free one (noalloc.cu): the tensor maps
// of one core-shape group and the per-phase GEMM group descriptors.
//
// One Newton-Schulz step (HyperParallel-FSDP section 2.3, Eq. (1)) runs as
// three launches over every group of a chunk: Gram A = X X^T, polynomial
// B' = b A + c A^2 + alpha I, apply Xt' = (a - alpha) Xt + Xt B'.  The
// iterate lives only as Xt = X^T ([n][m_pad] bf16 per matrix), ping-ponged
// between two buffers: step `it` reads Xt[it & 1] and writes Xt[(it + 1) & 1].
#include <cstdlib>
#include <mutex>

#include "muon_internal.h"

namespace muon {

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

int64_t cdiv64(int64_t a, int64_t b) { return (a + b - 1) / b; }

}  // namespace

bool encode_tiled(CUtensorMap* map, bool f32, const void* base, const uint64_t* dims,
                  const uint64_t* strides, const uint32_t* box, bool swizzle128) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[3] = {dims[0], dims[1], dims[2]};
  cuuint64_t st[2] = {strides[0], strides[1]};
  cuuint32_t b[3] = {box[0], box[1], box[2]};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
            const_cast<void*>(base), d, st, b, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool make_ns_map(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t cnt,
                 int64_t pitch, int64_t mstride, int box_rows) {
  const uint64_t dims[3] = {static_cast<uint64_t>(inner), static_cast<uint64_t>(rows),
                            static_cast<uint64_t>(cnt)};
  const uint64_t strides[2] = {static_cast<uint64_t>(pitch * 2),
                               static_cast<uint64_t>(mstride * 2)};
  const uint32_t box[3] = {static_cast<uint32_t>(gemm_block_k()),
                           static_cast<uint32_t>(box_rows), 1};
  return encode_tiled(map, false, base, dims, strides, box, true);
}

bool ns_group_maps(NsGroupDev& g) {
  const int bm = gemm_block_m(), bn = gemm_block_n();
  const int64_t xs = g.n * g.m_pad, as = g.m * g.m_pad;
  bool ok = true;
  for (int b = 0; b < 2; ++b) {
    // Gram: MN-major 64 (m) x 64 (n) chunks; apply: 128 rows (n) x 64 (m)
    ok = ok && make_ns_map(&g.map_gram[b], g.Xt[b], g.m, g.n, g.cnt, g.m_pad, xs, 64);
    ok = ok && make_ns_map(&g.map_xt[b], g.Xt[b], g.m, g.n, g.cnt, g.m_pad, xs, bm);
  }
  ok = ok && make_ns_map(&g.map_ap, g.A, g.m, g.m, g.cnt, g.m_pad, as, bm) &&
       make_ns_map(&g.map_aq, g.A, g.m, g.m, g.cnt, g.m_pad, as, bn) &&
       make_ns_map(&g.map_a64, g.A, g.m, g.m, g.cnt, g.m_pad, as, 64) &&
       make_ns_map(&g.map_bp, g.B, g.m, g.m, g.cnt, g.m_pad, as, bm) &&
       make_ns_map(&g.map_bq, g.B, g.m, g.m, g.cnt, g.m_pad, as, bn) &&
       make_ns_map(&g.map_b64, g.B, g.m, g.m, g.cnt, g.m_pad, as, 64);
  if (g.A_lo) {   // the same boxes on the lo halves
    for (int b = 0; b < 2; ++b) {
      ok = ok && make_ns_map(&g.lo_gram[b], g.Xt_lo[b], g.m, g.n, g.cnt, g.m_pad, xs, 64);
      ok = ok && make_ns_map(&g.lo_xt[b], g.Xt_lo[b], g.m, g.n, g.cnt, g.m_pad, xs, bm);
    }
    ok = ok && make_ns_map(&g.lo_ap, g.A_lo, g.m, g.m, g.cnt, g.m_pad, as, bm) &&
         make_ns_map(&g.lo_aq, g.A_lo, g.m, g.m, g.cnt, g.m_pad, as, bn) &&
         make_ns_map(&g.lo_a64, g.A_lo, g.m, g.m, g.cnt, g.m_pad, as, 64) &&
         make_ns_map(&g.lo_bp, g.B_lo, g.m, g.m, g.cnt, g.m_pad, as, bm) &&
         make_ns_map(&g.lo_bq, g.B_lo, g.m, g.m, g.cnt, g.m_pad, as, bn) &&
         make_ns_map(&g.lo_b64, g.B_lo, g.m, g.m, g.cnt, g.m_pad, as, 64);
  }
  return ok;
}

bool gemm_use_pair(int64_t tiles, int sms, int64_t min_m) {
  if (const char* v = std::getenv("MUON_GEMM_PAIR")) {
    if (v[0] == '0') return false;
    if (v[0] == '1') return true;
  }
  // Measured on one GB300, the same box back to back (ms per step, unpaired
  // -> paired): large sweep (m = 8192, 16384; power-capped, 1500 -> 1650
  // MHz) 520.2 -> 505.6; Llama-3-8B shapes (m <= 4096) 334.6 -> 337.4; MoE
  // experts (m = 768, full clocks) 6.14 -> 6.25.  Pairs move a third less
  // operand data per MMA, which buys clock under the power cap, but tie two
  // CTAs' pipelines together: only the largest core shapes gain.  They also
  // halve the number of work units, so a launch needs two waves of pairs.
  return min_m >= 8192 && tiles >= 4LL * sms;
}

bool gemm_use_wide(int epi, int64_t tiles, int sms, int min_kb, double mean_kb) {
  if (const char* v = std::getenv("MUON_GEMM_WIDE")) {
    if (v[0] == '0') return false;
    if (v[0] == '1') return true;
  }
  // Measured on one GB300, the same box back to back (ms per launch, single
  // tiles -> WIDE; the large sweep power-capped at 1590-1650 MHz): large
  // sweep (K >= 8192) Gram 3.00 -> 2.76, polynomial 2.28 -> 2.14, apply
  // 6.18 -> 5.49 (step 475 -> 432); Llama-3-8B shapes (mean K ~4000, k/v at
  // K = 1024) Gram 1.306 -> 1.238, apply 2.477 -> 2.323, polynomial 0.571 ->
  // 0.620; MoE experts (K = 768 / 2048) Gram 0.288 -> 0.302, polynomial
  // 0.158 -> 0.216, apply 0.478 -> 0.549.  A block needs both accumulators,
  // so its epilogue no longer overlaps the next block's MMAs: only long K
  // amortises that, and the polynomial (its epilogue loads the b A term and
  // writes the mirror too) needs the longest.
  if (tiles < 2LL * sms) return false;
  return epi == kEpiPoly ? min_kb >= 128 : mean_kb >= 48.0;
}

void ns_fill_group(GemmGroup& G, const NsGroupDev& g, int phase, int it, int tile_base,
                   bool pair, bool wide) {
  const bool pt = pair || wide;   // tiles are pair tiles
  const int bm = gemm_block_m(), bn = gemm_block_n(), bk = gemm_block_k();
  G.m = static_cast<int>(g.m);
  G.n = static_cast<int>(g.n);
  G.count = static_cast<int>(g.cnt);
  G.inv = g.inv;
  G.tile_base = tile_base;
  if (phase == kEpiGram) {
    G.mapA = g.map_gram[it & 1];
    G.mapB = g.map_gram[it & 1];
    G.mapC = g.map_ap;
    G.mapD = g.map_a64;
    if (g.A_lo) {
      G.mapAlo = G.mapBlo = g.lo_gram[it & 1];
      G.mapClo = g.lo_ap;
      G.mapDlo = g.lo_a64;
    }
    G.partial = g.partial;
    G.tile_cnt = g.tile_cnt;
    G.nt = static_cast<int>(cdiv64(g.m, bn));
    G.mt = static_cast<int>(cdiv64(g.m, bm));
    G.ksplit = g.ksplit;
    G.kb_per_split = g.kb_per_split;
    G.num_kb = g.num_kb_gram;
    G.tiles_per_mat = pt ? gemm_sym_pair_tiles(static_cast<int>(g.m))
                         : static_cast<int>(g.tri * g.ksplit);
  } else if (phase == kEpiPoly) {
    G.mapA = g.map_ap;      // operand rows and the epilogue's A tiles
    G.mapB = pair ? g.map_ap : g.map_aq;   // a pair loads B in 128-row halves
    G.mapC = g.map_bp;
    G.mapD = g.map_b64;
    if (g.A_lo) {
      G.mapAlo = g.lo_ap;
      G.mapBlo = g.lo_aq;
      G.mapClo = g.lo_bp;
      G.mapDlo = g.lo_b64;
    }
    G.nt = static_cast<int>(cdiv64(g.m, bn));
    G.mt = static_cast<int>(cdiv64(g.m, bm));
    G.ksplit = 1;
    G.num_kb = static_cast<int>(cdiv64(g.m, bk));
    G.kb_per_split = G.num_kb;
    G.tiles_per_mat = pt ? gemm_sym_pair_tiles(static_cast<int>(g.m)) : static_cast<int>(g.tri);
  } else {
    G.mapA = g.map_xt[it & 1];
    G.mapB = pair ? g.map_bp : g.map_bq;
    G.mapC = g.map_xt[(it + 1) & 1];
    if (g.A_lo) {
      G.mapAlo = g.lo_xt[it & 1];
      G.mapBlo = g.lo_bq;
      G.mapClo = g.lo_xt[(it + 1) & 1];
    }
    G.nt = static_cast<int>(cdiv64(g.m, bn));
    G.mt = static_cast<int>(cdiv64(g.n, bm));
    G.ksplit = 1;
    G.num_kb = static_cast<int>(cdiv64(g.m, bk));
    G.kb_per_split = G.num_kb;
    G.tiles_per_mat = G.nt * (pt ? (G.mt + 1) / 2 : G.mt);
  }
}

// ---- Gram-space NS --------------------------------------------------------------------
// DMuon-2 Appendix C.3: every step multiplies X by a polynomial of its Gram
// matrix, so with R_0 = X0 X0^T / ||X0||^2 the iteration runs on m x m
// matrices: B'_k = b R_k + c R_k^2 + alpha I, T = (a - alpha) R_k + R_k B'_k,
// R_{k+1} = (a - alpha) T + T B'_k, Q_{k+1} = (a - alpha) Q_k + Q_k B'_k
// (Q_1 = P_0 = a I + b R_0 + c R_0^2), and O = Q_K X0 / ||X0|| at the end.
// All of R, T, B', Q are polynomials of R_0, so their products are
// symmetric: each runs on the polynomial kernel (upper tiles plus mirror),
// whose epilogue b' A + c' (A B) + alpha' I gives the shifted forms with
// b' = a - alpha, c' = 1, alpha' = 0.  The B operand is read MN-major (A B,
// not A B^T): the tiles that cross the diagonal are stored as computed, so
// the rounded T, R and Q carry a small antisymmetric part, and products with
// the transpose would multiply that part by about q(l) (a - b l + c l^2)
// (~7 for the default quintic at l = 1) every step instead of damping it.
// The iteration restarts every few steps (the section's mid-way restart):
// X_k = Q X is formed by one apply, R is recomputed as the Gram of X_k, and Q
// starts again from P_k.  Without it, bf16 R loses the small eigenvalues of
// an ill-conditioned X (R squares its condition number) and Q's growing
// range amplifies that loss.

bool ns_gs_maps(NsGroupDev& g) {
  const int bm = gemm_block_m();
  const int64_t as = g.m * g.m_pad;
  bool ok = true;
  for (int i = 0; i < 5; ++i)
    ok = ok && make_ns_map(&g.s_p[i], g.S[i], g.m, g.m, g.cnt, g.m_pad, as, bm) &&
         make_ns_map(&g.s_64[i], g.S[i], g.m, g.m, g.cnt, g.m_pad, as, 64);
  return ok;
}

void ns_fill_gs_gram(GemmGroup& G, const NsGroupDev& g, int src, int tile_base, bool pair,
                     bool wide) {
  ns_fill_group(G, g, kEpiGram, src, tile_base, pair, wide);   // reads Xt[src]
  G.mapC = g.s_p[kGsR];
  G.mapD = g.s_64[kGsR];
}

void ns_fill_gs_sym(GemmGroup& G, const NsGroupDev& g, int a, int b, int c, int tile_base,
                    bool pair, bool wide) {
  ns_fill_group(G, g, kEpiPoly, 0, tile_base, pair, wide);
  G.mapA = g.s_p[a];                       // operand rows and the epilogue's b' S[a] tiles
  G.mapB = g.s_64[b];                      // MN-major 64 x 64 chunks (also for pairs)
  G.mapC = g.s_p[c];
  G.mapD = g.s_64[c];
}

void ns_fill_gs_apply(GemmGroup& G, const NsGroupDev& g, int q, int src, int tile_base,
                      bool pair, bool wide) {
  ns_fill_group(G, g, kEpiApply, src, tile_base, pair, wide);   // reads Xt[src], writes Xt[src ^ 1]
  G.mapB = g.s_64[q];                      // Xt Q, Q read MN-major
}

}  // namespace muon
