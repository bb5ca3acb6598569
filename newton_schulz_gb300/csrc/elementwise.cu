// Memory-bound kernels of the Muon step.
//
//  prep_kernel   (K1)  momentum + Nesterov, per-matrix ||D||_F^2 partials,
//                      bf16 cast into the Newton-Schulz workspace layout
//                      Xt = X^T ([n][m]: the stored layout when rows > cols,
//                      else the transpose), in one pass over G and Mom.
//                      DMuon-2 section 2.1 (M_t = mu*M_{t-1} + G, Nesterov);
//                      HyperParallel-FSDP section 2.3 Eq. (1) (X0 = G/(||G||+eps))
//                      and section 6.6 (transpose-first, bf16 NS path).
//  finish_kernel (K6)  W <- (1 - lr*wd)*W - lr*s*O (RFC issue 204 item 6,
//                      DMuon-2 section 2.1), or the copy-back of an NS-only call;
//                      O is read from Xt, through a shared-memory transpose
//                      when the stored layout is [m][n].  finish_tall_kernel
//                      is the same update in two row passes a thread, for
//                      launches whose weights are all bf16.
//
// All are HBM-bound streaming kernels: 16-byte vector loads and stores,
// warp-shuffle reductions, deterministic two-stage norm (per-tile partials,
// then the last-arriving block of each matrix sums them in a fixed order).
#include "muon_internal.h"

namespace muon {

namespace {

__device__ __forceinline__ float bf16_to_f(__nv_bfloat16 v) { return __bfloat162float(v); }

__device__ __forceinline__ void store8_f32(float* p, const float* d) {
  *reinterpret_cast<float4*>(p) = make_float4(d[0], d[1], d[2], d[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(d[4], d[5], d[6], d[7]);
}

// Raw 16-byte loads are kept apart from their conversions so that a thread
// issues all of its loads before the first conversion waits for data.
__device__ __forceinline__ void unpack8_bf16(uint4 u, float* d) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float2 f = __bfloat1622float2(h[j]);
    d[2 * j] = f.x;
    d[2 * j + 1] = f.y;
  }
}

__device__ __forceinline__ void unpack4_f32(uint4 u, float* d) {
  d[0] = __uint_as_float(u.x);
  d[1] = __uint_as_float(u.y);
  d[2] = __uint_as_float(u.z);
  d[3] = __uint_as_float(u.w);
}

__device__ __forceinline__ void load8_bf16(const __nv_bfloat16* p, float* d) {
  unpack8_bf16(*reinterpret_cast<const uint4*>(p), d);
}

__device__ __forceinline__ uint4 pack8_bf16(const float* d) {
  uint4 u;
  __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
  for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(d[2 * j], d[2 * j + 1]);
  return u;
}

// lo = bf16(d - bf16(d)): the second half of a split bf16 pair
__device__ __forceinline__ uint4 pack8_bf16_lo(const float* d) {
  float r[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) r[j] = d[j] - __bfloat162float(__float2bfloat16_rn(d[j]));
  return pack8_bf16(r);
}

// The slice that block `blk` belongs to: the last one whose first block is
// at or before it.  The launch's first-block table is read into shared memory
// by the block's threads in parallel (indexed reads of the parameter block
// are generic loads; a scan would chain one per slice), then searched there.
// Every thread of the block must call it (it holds a barrier).
template <typename Slice>
__device__ __forceinline__ int find_slice(const Slice* s, int n, int blk) {
  __shared__ int base[kMaxSlices];
  for (int i = threadIdx.x; i < n; i += blockDim.x) base[i] = s[i].tile_base;
  __syncthreads();
  int lo = 0, hi = n - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (base[mid] <= blk) lo = mid;
    else hi = mid - 1;
  }
  return lo;
}

// Column of element (r, c) of the prep kernel's 64 x 64 fp32 tile (pitch 65):
// an XOR of bits 2..4 of c with bits 3..5 of r and of c, which leaves each of
// the tile's access patterns -- 8-wide row writes, 8-deep column reads and
// 16-wide row or column reads for the norm -- one wavefront per warp
// instruction (a bijection within each row; checked exhaustively on the host).
__device__ __forceinline__ int prep_col(int r, int c) { return c ^ ((((r >> 3) ^ (c >> 3)) & 7) << 2); }

}  // namespace

// ---------------------------------------------------------------------------
// K1
// ---------------------------------------------------------------------------
// Six resident blocks per SM (at most 40 registers a thread): the loads in
// flight per SM set this kernel's rate (48 registers, five blocks, measured
// slower).
__global__ void __launch_bounds__(256, 6) prep_kernel(const __grid_constant__ PrepParams p) {
  // fp32 tile of D in the stored [r][c] layout (+1 pad against bank conflicts)
  __shared__ float sD[kPrepTile][kPrepTile + 1];
  __shared__ float red[8];
  __shared__ double dred[256];
  __shared__ int s_last;

  const int si = find_slice(p.s, p.n_slices, blockIdx.x);
  const PrepSlice& s = p.s[si];
  const int local = blockIdx.x - s.tile_base;
  const int tiles = s.tiles_r * s.tiles_c;
  const int mat = local / tiles;
  const int t = local - mat * tiles;
  const int ti = t / s.tiles_c, tj = t - ti * s.tiles_c;
  const int64_t r0 = (int64_t)ti * kPrepTile, c0 = (int64_t)tj * kPrepTile;
  const int tx = threadIdx.x & 7, ty = threadIdx.x >> 3;
  const int64_t moff = (int64_t)mat * s.r * s.c;

#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int lr = ty + 32 * pass;
    const int64_t gr = r0 + lr;
    const int lc = tx * 8;
    const int64_t gc = c0 + lc;
    float d[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) d[j] = 0.f;
    int nvalid = 0;
    if (gr < s.r && gc < s.c) nvalid = (int)min((int64_t)8, s.c - gc);
    // debug builds: the element range lies in the slice's tensors
    if (nvalid > 0 && !dbg_ok(mat < s.count && moff + gr * s.c + gc + nvalid <= (int64_t)s.count * s.r * s.c,
                              p.status))
      nvalid = 0;
    if (nvalid > 0) {
      const int64_t e = moff + gr * s.c + gc;
      const bool v8 = nvalid == 8 && s.vec;
      float g[8], m[8];
      if (v8) {
        // G's and Mom's raw bits first, then the conversions: a bf16 G
        // converted next to its load would hold Mom's load back until G came
        uint4 g0, g1 = make_uint4(0u, 0u, 0u, 0u), m0 = g1, m1 = g1;
        if (s.g_dtype == 0) {
          const uint4* g4 = reinterpret_cast<const uint4*>(static_cast<const float*>(s.G) + e);
          g0 = __ldcs(g4);
          g1 = __ldcs(g4 + 1);
        } else {
          g0 = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(s.G) + e);
        }
        if (p.step_mode) {
          const uint4* m4 = reinterpret_cast<const uint4*>(s.Mom + e);
          m0 = __ldcs(m4);
          m1 = __ldcs(m4 + 1);
        }
        if (s.g_dtype == 0) {
          unpack4_f32(g0, g);
          unpack4_f32(g1, g + 4);
        } else {
          unpack8_bf16(g0, g);
        }
        unpack4_f32(m0, m);
        unpack4_f32(m1, m + 4);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          g[j] = 0.f;
          if (j < nvalid)
            g[j] = s.g_dtype == 0 ? reinterpret_cast<const float*>(s.G)[e + j]
                                  : bf16_to_f(reinterpret_cast<const __nv_bfloat16*>(s.G)[e + j]);
        }
        if (p.step_mode) {
#pragma unroll
          for (int j = 0; j < 8; ++j) m[j] = j < nvalid ? s.Mom[e + j] : 0.f;
        }
      }
      if (p.step_mode) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float mn = fmaf(p.mu, m[j], g[j]);          // M_t = mu*M_{t-1} + G
          m[j] = mn;
          d[j] = p.nesterov ? fmaf(p.mu, mn, g[j]) : mn;    // D = G + mu*M_t
        }
        if (v8) {
          store8_f32(s.Mom + e, m);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            if (j < nvalid) s.Mom[e + j] = m[j];
        }
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) d[j] = g[j];
      }
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j >= nvalid) d[j] = 0.f;
      // [r][c] copy: the padded workspace row always has room for 8 elements.
      if (s.direct && dbg_ok(gc + 8 <= s.pitch_d, p.status)) {
        const int64_t o = (int64_t)mat * s.mstride_d + gr * s.pitch_d + gc;
        *reinterpret_cast<uint4*>(s.direct + o) = pack8_bf16(d);
        if (s.direct_lo) *reinterpret_cast<uint4*>(s.direct_lo + o) = pack8_bf16_lo(d);
      }
    }
#pragma unroll
    for (int j = 0; j < 8; ++j) sD[lr][prep_col(lr, lc + j)] = d[j];
  }
  __syncthreads();
  // [c][r] copy from the shared-memory tile.
#pragma unroll
  for (int pass = 0; pass < 2; ++pass) {
    const int lcc = ty + 32 * pass;
    const int64_t gcc = c0 + lcc;
    const int lrr = tx * 8;
    const int64_t grr = r0 + lrr;
    if (s.transp && gcc < s.c && grr < s.r && dbg_ok(grr + 8 <= s.pitch_t, p.status)) {
      float v[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) v[j] = sD[lrr + j][prep_col(lrr + j, lcc)];
      const int64_t o = (int64_t)mat * s.mstride_t + gcc * s.pitch_t + grr;
      *reinterpret_cast<uint4*>(s.transp + o) = pack8_bf16(v);
      if (s.transp_lo) *reinterpret_cast<uint4*>(s.transp_lo + o) = pack8_bf16_lo(v);
    }
  }

  // Tile partial of ||D||_F^2, summed in an order fixed by the coordinates of
  // the NS operand X (X = D, or D^T when transposed), so that a matrix and its
  // transpose give bit-identical norms.  Thread t sums 16 consecutive X
  // columns of X row t/4; then a fixed shuffle tree and the 8 warps in order.
  float ssq = 0.f;
  {
    const int xi = threadIdx.x >> 2, xj0 = (threadIdx.x & 3) * 16;
#pragma unroll
    for (int j = 0; j < 16; ++j) {
      const float v = s.trans ? sD[xj0 + j][prep_col(xj0 + j, xi)] : sD[xi][prep_col(xi, xj0 + j)];
      ssq = fmaf(v, v, ssq);
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = ssq;
  __syncthreads();
  if (threadIdx.x == 0) {
    float b = 0.f;
    for (int w = 0; w < 8; ++w) b += red[w];
    // partial slot indexed by the X tile coordinates
    const int xt = s.trans ? tj * s.tiles_r + ti : ti * s.tiles_c + tj;
    s.ssq_part[(int64_t)mat * tiles + xt] = b;
    __threadfence();
    const unsigned prev = atomicAdd(&s.cnt[mat], 1u);
    s_last = (prev == (unsigned)(tiles - 1));
  }
  __syncthreads();
  if (!s_last) return;
  // Last block of this matrix: sum the partials in a fixed order.
  __threadfence();
  double acc = 0.0;
  const float* part = s.ssq_part + (int64_t)mat * tiles;
  for (int i = threadIdx.x; i < tiles; i += 256) acc += (double)__ldcg(part + i);
  dred[threadIdx.x] = acc;
  __syncthreads();
  for (int w = 128; w > 0; w >>= 1) {
    if (threadIdx.x < w) dred[threadIdx.x] += dred[threadIdx.x + w];
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    const double tot = dred[0];
    const double nrm = sqrt(tot);
    if (!isfinite(tot)) atomicOr(p.status, kDevNonfinite);
    s.inv[mat] = (float)(1.0 / (nrm + (double)p.eps));
    s.cnt[mat] = 0u;
  }
}

// ---------------------------------------------------------------------------
// K6
// ---------------------------------------------------------------------------
// One row pass, 8 elements a thread; eight resident blocks per SM (at most
// 32 registers a thread: the W and O loads in flight per SM set the rate on
// fp32 weights).  On bf16 weights it is issue-bound, and launches whose
// weights are all bf16 run finish_tall_kernel instead.
__global__ void __launch_bounds__(256, 8) finish_kernel(const __grid_constant__ FinParams p) {
  // o_trans tiles: the O tile [kFinTRows][kFinTCols] (fp32: hi + lo in the
  // high-precision mode), transposed from Xt on the way in; the odd pitch
  // (65 words) keeps the scattered writes free of bank conflicts
  __shared__ __align__(16) float sO[kFinTRows][kFinTCols + 1];
  const int si = find_slice(p.s, p.n_slices, blockIdx.x);
  const FinSlice& s = p.s[si];
  const int local = blockIdx.x - s.tile_base;
  const int tiles = s.tiles_r * s.tiles_c;
  const int mat = local / tiles;
  const int t = local - mat * tiles;
  const int ti = t / s.tiles_c, tj = t - ti * s.tiles_c;
  // the thread's elements of W: row gr, columns [gc, gc + nvalid)
  int64_t gr, gc;
  if (s.o_trans) {
    gr = (int64_t)ti * kFinTRows + (threadIdx.x >> 3);
    gc = (int64_t)tj * kFinTCols + (threadIdx.x & 7) * 8;
  } else {
    gr = (int64_t)ti * kFinRows + (threadIdx.x >> 5);
    gc = (int64_t)tj * kFinCols + (threadIdx.x & 31) * 8;
  }
  const bool live = gr < s.r && gc < s.c;
  const int nvalid = live ? (int)min((int64_t)8, s.c - gc) : 0;
  const int64_t e = (int64_t)mat * s.r * s.c + gr * s.c + gc;
  // debug builds: the element range lies in the slice's W
  const bool w_ok =
      live && dbg_ok(mat < s.count && e + nvalid <= (int64_t)s.count * s.r * s.c, p.status);
  const bool vec8 = w_ok && nvalid == 8 && s.vec;
  // A full vector of W is loaded first, as raw bits, and converted only once
  // O is in registers: the two loads' latencies overlap instead of adding up
  // (a conversion next to its load would make the thread wait for W there).
  uint4 wr0 = make_uint4(0u, 0u, 0u, 0u), wr1 = wr0;
  if (p.step_mode && vec8) {
    if (s.w_dtype == 0) {
      const uint4* w4 = reinterpret_cast<const uint4*>(static_cast<const float*>(s.W) + e);
      wr0 = __ldcs(w4);
      wr1 = __ldcs(w4 + 1);
    } else {
      wr0 = *reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(s.W) + e);
    }
  }
  float o[8];
  if (s.o_trans) {
    // O[gr][gc] = Xt[gc][gr]: each thread brings 8 consecutive gr of one Xt
    // row (a 64-byte segment per 4 threads), then reads 8 consecutive gc
    const int64_t r0 = (int64_t)ti * kFinTRows, c0 = (int64_t)tj * kFinTCols;
    {
      const int lc = threadIdx.x >> 2, q = threadIdx.x & 3;
      const int64_t xr = c0 + lc, xc = r0 + 8 * q;
      float f[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] = 0.f;
      // (the loads below touch [xc, min(xc + 8, r)) of the row)
      if (xr < s.c && dbg_ok(mat < s.count && min(xc + 8, s.r) <= s.pitch_o, p.status)) {
        const int64_t oo = (int64_t)mat * s.mstride_o + xr * s.pitch_o + xc;
        if (xc + 8 <= s.r) {
          load8_bf16(s.O + oo, f);
          if (s.O_lo) {
            float l[8];
            load8_bf16(s.O_lo + oo, l);
#pragma unroll
            for (int j = 0; j < 8; ++j) f[j] += l[j];
          }
        } else {
          for (int j = 0; j < 8; ++j)
            if (xc + j < s.r) f[j] = bf16_to_f(s.O[oo + j]) + (s.O_lo ? bf16_to_f(s.O_lo[oo + j]) : 0.f);
        }
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) sO[8 * q + j][lc] = f[j];
    }
    __syncthreads();
    const int lr = threadIdx.x >> 3, lc0 = (threadIdx.x & 7) * 8;
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = sO[lr][lc0 + j];
  } else {
    // both halves' raw bits first, then the conversions
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] = 0.f;
    if (live && dbg_ok(mat < s.count && gc + 8 <= s.pitch_o, p.status)) {
      const int64_t oo = (int64_t)mat * s.mstride_o + gr * s.pitch_o + gc;
      const uint4 hi = *reinterpret_cast<const uint4*>(s.O + oo);
      uint4 lo = make_uint4(0u, 0u, 0u, 0u);
      if (s.O_lo) lo = *reinterpret_cast<const uint4*>(s.O_lo + oo);
      unpack8_bf16(hi, o);
      if (s.O_lo) {
        float l[8];
        unpack8_bf16(lo, l);
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] += l[j];
      }
    }
  }
  if (!w_ok) return;

  const float os = s.inv ? s.inv[mat] : 1.f;

  if (p.step_mode) {
    const float decay = 1.f - p.lr * p.wd;
    const float step = p.lr * s.scale * os;
    float w[8];
    if (s.w_dtype == 0) {
      float* W = reinterpret_cast<float*>(s.W);
      if (vec8) {
        unpack4_f32(wr0, w);
        unpack4_f32(wr1, w + 4);
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = fmaf(decay, w[j], -step * o[j]);
        store8_f32(W + e, w);
      } else {
        for (int j = 0; j < nvalid; ++j) W[e + j] = fmaf(decay, W[e + j], -step * o[j]);
      }
    } else {
      __nv_bfloat16* W = reinterpret_cast<__nv_bfloat16*>(s.W);
      if (vec8) {
        unpack8_bf16(wr0, w);
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = fmaf(decay, w[j], -step * o[j]);
        *reinterpret_cast<uint4*>(W + e) = pack8_bf16(w);
      } else {
        for (int j = 0; j < nvalid; ++j)
          W[e + j] = __float2bfloat16_rn(fmaf(decay, bf16_to_f(W[e + j]), -step * o[j]));
      }
    }
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j) o[j] *= os;
    if (s.w_dtype == 0) {
      float* W = reinterpret_cast<float*>(s.W);
      if (vec8) store8_f32(W + e, o);
      else for (int j = 0; j < nvalid; ++j) W[e + j] = o[j];
    } else {
      __nv_bfloat16* W = reinterpret_cast<__nv_bfloat16*>(s.W);
      if (vec8) *reinterpret_cast<uint4*>(W + e) = pack8_bf16(o);
      else for (int j = 0; j < nvalid; ++j) W[e + j] = __float2bfloat16_rn(o[j]);
    }
  }
}

// Update of a launch whose weights are all bf16 (6 bytes moved per element):
// tiles twice as tall as finish_kernel's, two row passes a thread (16
// elements), so that a block's fixed costs (the slice lookup, the index
// arithmetic, the transposed tile's barrier) and its bytes in flight match
// those of an fp32 launch (10 bytes per element) at one pass.  Same
// arithmetic as finish_kernel; all four 16-byte loads (W and O, both passes)
// are issued before the first conversion.  56 registers a thread, four
// resident blocks per SM: capped at 48 registers (five blocks) the kernel
// spills and measured 0.64 of HBM against 0.77-0.79 uncapped, on 8
// Llama-3-8B layers, where the one-pass kernel is issue-bound at 0.63.
__global__ void __launch_bounds__(256) finish_tall_kernel(const __grid_constant__ FinParams p) {
  __shared__ __align__(16) float sO[2 * kFinTRows][kFinTCols + 1];
  const int si = find_slice(p.s, p.n_slices, blockIdx.x);
  const FinSlice& s = p.s[si];
  const int local = blockIdx.x - s.tile_base;
  const int tiles = s.tiles_r * s.tiles_c;
  const int mat = local / tiles;
  const int t = local - mat * tiles;
  const int ti = t / s.tiles_c, tj = t - ti * s.tiles_c;
  const bool tr = s.o_trans != 0;
  const int rstep = tr ? kFinTRows : kFinRows;             // rows between the two passes
  // the thread's W elements: rows gr and gr + rstep, columns [gc, gc + nvalid)
  const int64_t gr = (int64_t)ti * (2 * rstep) + (tr ? threadIdx.x >> 3 : threadIdx.x >> 5);
  const int64_t gc = tr ? (int64_t)tj * kFinTCols + (threadIdx.x & 7) * 8
                        : (int64_t)tj * kFinCols + (threadIdx.x & 31) * 8;
  const int nvalid = gc < s.c ? (int)min((int64_t)8, s.c - gc) : 0;
  const int64_t e = (int64_t)mat * s.r * s.c + gr * s.c + gc;
  const int64_t wstep = (int64_t)rstep * s.c;
  const int64_t wtotal = (int64_t)s.count * s.r * s.c;
  // debug builds: each pass's element range lies in the slice's bf16 W
  const bool ok0 = gr < s.r && nvalid > 0 &&
                   dbg_ok(s.w_dtype != 0 && mat < s.count && e + nvalid <= wtotal, p.status);
  const bool ok1 = gr + rstep < s.r && nvalid > 0 &&
                   dbg_ok(s.w_dtype != 0 && mat < s.count && e + wstep + nvalid <= wtotal, p.status);
  const bool v8 = nvalid == 8 && s.vec;
  __nv_bfloat16* W = static_cast<__nv_bfloat16*>(s.W) + e;
  uint4 w0 = make_uint4(0u, 0u, 0u, 0u), w1 = w0, o0 = w0, o1 = w0;
  if (p.step_mode && v8) {
    if (ok0) w0 = *reinterpret_cast<const uint4*>(W);
    if (ok1) w1 = *reinterpret_cast<const uint4*>(W + wstep);
  }
  // O's hi half as raw bits at the thread's load positions (the
  // high-precision lo half is added when the hi half is converted)
  const int lc = threadIdx.x >> 2, q = threadIdx.x & 3;     // transposed loads: Xt row, 8-chunk
  const int64_t xr = (int64_t)tj * kFinTCols + lc, xc = (int64_t)ti * (2 * kFinTRows) + 8 * q;
  const int64_t ooff = tr ? (int64_t)mat * s.mstride_o + xr * s.pitch_o + xc
                          : (int64_t)mat * s.mstride_o + gr * s.pitch_o + gc;
  const int64_t ostep = tr ? kFinTRows : (int64_t)rstep * s.pitch_o;
  const bool of0 = tr ? (xr < s.c && xc + 8 <= s.r &&
                         dbg_ok(mat < s.count && xc + 8 <= s.pitch_o, p.status))
                      : (ok0 && dbg_ok(gc + 8 <= s.pitch_o, p.status));
  const bool of1 = tr ? (xr < s.c && xc + kFinTRows + 8 <= s.r &&
                         dbg_ok(mat < s.count && xc + kFinTRows + 8 <= s.pitch_o, p.status))
                      : (ok1 && dbg_ok(gc + 8 <= s.pitch_o, p.status));
  if (of0) o0 = *reinterpret_cast<const uint4*>(s.O + ooff);
  if (of1) o1 = *reinterpret_cast<const uint4*>(s.O + ooff + ostep);
  float o[8];
  if (tr) {
    // O[gr][gc] = Xt[gc][gr], staged through the [2 kFinTRows][kFinTCols]
    // tile (odd pitch: the scattered writes are free of bank conflicts)
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 raw = h ? o1 : o0;
      const bool full = h ? of1 : of0;
      const int64_t xch = xc + h * kFinTRows;
      float f[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) f[j] = 0.f;
      if (full) {
        unpack8_bf16(raw, f);
        if (s.O_lo) {
          float l[8];
          load8_bf16(s.O_lo + ooff + h * ostep, l);
#pragma unroll
          for (int j = 0; j < 8; ++j) f[j] += l[j];
        }
      } else if (xr < s.c && xch < s.r && dbg_ok(mat < s.count && s.r <= s.pitch_o, p.status)) {
        // (touches [xch, r) of the row, fewer than 8 elements)
        const int64_t oo = ooff + h * ostep;
        for (int j = 0; j < 8; ++j)
          if (xch + j < s.r) f[j] = bf16_to_f(s.O[oo + j]) + (s.O_lo ? bf16_to_f(s.O_lo[oo + j]) : 0.f);
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) sO[h * kFinTRows + 8 * q + j][lc] = f[j];
    }
    __syncthreads();
  }
  const float os = s.inv ? s.inv[mat] : 1.f;
  const float decay = 1.f - p.lr * p.wd;
  const float step = p.lr * s.scale * os;
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    if (!(h ? ok1 : ok0)) continue;
    __nv_bfloat16* Wh = W + h * wstep;
    if (tr) {
      const int lr = threadIdx.x >> 3, lc0 = (threadIdx.x & 7) * 8;
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j] = sO[h * kFinTRows + lr][lc0 + j];
    } else {
      unpack8_bf16(h ? o1 : o0, o);
      if (s.O_lo && (h ? of1 : of0)) {
        float l[8];
        load8_bf16(s.O_lo + ooff + h * ostep, l);
#pragma unroll
        for (int j = 0; j < 8; ++j) o[j] += l[j];
      }
    }
    if (p.step_mode) {
      if (v8) {
        float w[8];
        unpack8_bf16(h ? w1 : w0, w);
#pragma unroll
        for (int j = 0; j < 8; ++j) w[j] = fmaf(decay, w[j], -step * o[j]);
        *reinterpret_cast<uint4*>(Wh) = pack8_bf16(w);
      } else {
        for (int j = 0; j < nvalid; ++j)
          Wh[j] = __float2bfloat16_rn(fmaf(decay, bf16_to_f(Wh[j]), -step * o[j]));
      }
    } else {
#pragma unroll
      for (int j = 0; j < 8; ++j) o[j] *= os;
      if (v8) *reinterpret_cast<uint4*>(Wh) = pack8_bf16(o);
      else for (int j = 0; j < nvalid; ++j) Wh[j] = __float2bfloat16_rn(o[j]);
    }
  }
}

// ---------------------------------------------------------------------------
// Guard mode: count the bytes of each band (one block per band) that differ
// from the fill pattern.
// ---------------------------------------------------------------------------
__global__ void __launch_bounds__(256) guard_check_kernel(const __grid_constant__ GuardParams p) {
  const uint4* band = reinterpret_cast<const uint4*>(p.base + p.off[blockIdx.x]);
  const unsigned pat = p.pattern * 0x01010101u;
  unsigned bad = 0;
  for (unsigned i = threadIdx.x; i < p.bytes / 16; i += blockDim.x) {
    const uint4 v = __ldcg(band + i);
    const unsigned w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const unsigned d = w[k] ^ pat;
#pragma unroll
      for (int b = 0; b < 4; ++b) bad += ((d >> (8 * b)) & 0xffu) ? 1u : 0u;
    }
  }
  if (bad) atomicAdd(p.bad, static_cast<unsigned long long>(bad));
}

cudaError_t launch_guard_check(const GuardParams& p, cudaStream_t s) {
  if (p.n <= 0) return cudaSuccess;
  guard_check_kernel<<<p.n, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_prep(const PrepParams& p, cudaStream_t s) {
  if (p.total_blocks <= 0) return cudaSuccess;
  prep_kernel<<<p.total_blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_finish(const FinParams& p, cudaStream_t s) {
  if (p.total_blocks <= 0) return cudaSuccess;
  if (p.passes == 2) finish_tall_kernel<<<p.total_blocks, 256, 0, s>>>(p);
  else finish_kernel<<<p.total_blocks, 256, 0, s>>>(p);
  return cudaGetLastError();
}

}  // namespace muon
