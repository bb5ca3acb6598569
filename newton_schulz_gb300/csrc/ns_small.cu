// Fused Muon step for core shapes with a small side (m <= 64 after the
// transpose-first rule): Gram-space Newton-Schulz in one persistent launch.
//
// Every NS step left-multiplies X by a polynomial of its Gram matrix, so the
// iteration can run on the m x m Gram matrix and multiply back into X once at
// the end; in exact arithmetic this equals the X-space iteration of the Muon
// page (DMuon-2, Appendix C.3 "Gram Newton-Schulz and Its Fast Kernels"):
//   R_0 = X0 X0^T / ||X0||_F^2,   P_k = a_k I + b_k R_k + c_k R_k^2,
//   R_{k+1} = P_k R_k P_k,        Q = P_{K-1} ... P_1 P_0,
//   O = Q X0 / ||X0||_F.
// R, P and Q stay fp32 (m <= 64: 17 products of m x m per matrix, on CUDA
// cores); X0 is bf16 and Q is applied as two bf16 operands Q = hi + lo, so
// rounding X0 to bf16 is the only bf16 step of the iteration.
//
// A work item is (matrix, block of wb columns of X).  One cooperative launch,
// one CTA per SM, every CTA resident; the CTA is warp-specialised:
//   warp 0      producer: TMA tile loads of G/Mom (first phase) and W (second
//               phase) into a ring of shared-memory stages, bulk copies of
//               the X0 tiles and Q images for the second phase;
//   warp 1      allocates TMEM and issues the tcgen05 MMAs;
//   warps 2..9  consumers: momentum, X0 and the epilogues.
// Phase 1, per stage (a range of columns of one item): M' = mu M + G (written
// back), D = G + mu M' (Nesterov) or M', X0 = bf16(D) written both to the
// stage's 128-byte-swizzled X0 tile and to the matrix's X0 image in the
// workspace; the MMA warp accumulates the item's Gram X0_blk X0_blk^T (fp32,
// TMEM, two 64-column chunks stacked as one 2m-row operand) stage by stage.
// The item's Gram is read back one stage into the next item, so its last
// MMAs overlap that stage.  The CTA whose item arrives last for a matrix sums the
// partials in block order, normalises by the trace (= ||X0||_F^2), runs the
// Gram-space steps and publishes Q.
// Phase 2, per item: wait for the matrix's Q, bulk-load Q (hi rows, then lo
// rows); per 128-column tile the producer brings the W tile (TMA) and the X0
// tile (bulk copy from the image), and the MMA warp forms O = Q X0 (A =
// MN-major view of X0, M = 128 columns, K = m; B = [Q_hi; Q_lo], N = 2 nmm)
// into the stage's TMEM slot; the consumers write W' = (1 - lr wd) W - lr s O
// (or O itself) from TMEM, summing the hi and lo halves.
// Arrival counters carry a per-launch epoch tag, so a launch never depends on
// what an earlier (possibly aborted) launch left in them.  Every wait is
// bounded; a timeout sets a status bit and the CTA's abort flag, after which
// every role runs to the end without waiting and no output is written.
#include "muon_internal.h"
#include "sm100_ptx.cuh"

namespace muon {

namespace {

constexpr int kT = kSmallCons;      // consumer threads
constexpr int kSets = kT / 128;     // consumer warp sets (4 warps cover the 128 TMEM lanes)
constexpr uint32_t kConsBar = 1;   // named barrier of the consumer warps

// Shared-memory control block: mbarriers, the TMEM slot and CTA flags.
struct SmallBars {
  uint64_t ring_full[kSmallMaxStages], cons_done[kSmallMaxStages], mma_done[kSmallMaxStages];
  uint64_t gram_full[2], q_full[2], q_free[2];
  uint64_t mma_fin;    // the MMA issuer's last MMAs have completed
  uint64_t st_w[kSmallMaxStages];   // second phase, TMA-store epilogue: the owning
                                    // set's 4 warps wrote the stage's W' tile
  uint32_t tslot;
  int last;
  int abort;
  int desc[kSmallMaxStages][4];      // per stage: kind, item (-1: none), first X column, flags
  int cur_item;      // first phase: the consumers' current item (-2: abort)
};

// the planner reserves 512 bytes for the control block (SmallParams::off_bar)
static_assert(sizeof(SmallBars) <= 512, "control block larger than its reserved space");

struct Ctx {
  SmallBars* B;
  unsigned* status;
  unsigned long long timeout_ns;
};

// Bounded mbarrier wait.  False on timeout (which sets the status bit and the
// CTA's abort flag) or once another role of the CTA has aborted.
__device__ bool mwait(uint64_t* bar, uint32_t parity, const Ctx& c) {
  const uint32_t addr = ptx::smem_u32(bar);
  if (ptx::mbar_try_wait(addr, parity)) return true;
  volatile int* ab = &c.B->abort;
  if (*ab) return false;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (it > 4) __nanosleep(64);   // leave issue slots to the working warps
    if (ptx::mbar_try_wait(addr, parity)) return true;
    if ((it & 63u) == 0) {
      if (*ab) return false;
      if (ptx::globaltimer() - t0 > c.timeout_ns) {
        atomicOr(c.status, kDevTimeout);
        *ab = 1;
        return false;
      }
    }
  }
}

// Bounded wait that ignores the abort flag: at the end of a role, for copies
// or MMAs still in flight (they finish whatever else happened).  A timeout
// only sets the status bit.
__device__ void mwait_drain(uint64_t* bar, uint32_t parity, const Ctx& c) {
  const uint32_t addr = ptx::smem_u32(bar);
  if (ptx::mbar_try_wait(addr, parity)) return;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(64);
    if (ptx::mbar_try_wait(addr, parity)) return;
    if ((it & 63u) == 0 && ptx::globaltimer() - t0 > c.timeout_ns) {
      atomicOr(c.status, kDevTimeout);
      return;
    }
  }
}

// Bounded wait for the phase a token from this thread's own arrival names
// (the token fixes the phase, so no parity has to be tracked).
__device__ bool mwait_token(uint64_t* bar, uint64_t tok, const Ctx& c) {
  const uint32_t addr = ptx::smem_u32(bar);
  if (ptx::mbar_try_wait_token(addr, tok)) return true;
  volatile int* ab = &c.B->abort;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait_token(addr, tok)) return true;
    if ((it & 63u) == 0) {
      if (*ab) return false;
      if (ptx::globaltimer() - t0 > c.timeout_ns) {
        atomicOr(c.status, kDevTimeout);
        *ab = 1;
        return false;
      }
    }
  }
}

// The same wait made once per warp (lane 0 polls), result broadcast.
__device__ __forceinline__ bool mwait_warp(uint64_t* bar, uint32_t parity, const Ctx& c) {
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = mwait(bar, parity, c) ? 1 : 0;
  return __shfl_sync(0xffffffffu, ok, 0) != 0;
}

__device__ __forceinline__ unsigned long long ld_acquire_u64(const unsigned long long* p) {
  unsigned long long v;
  asm volatile("ld.acquire.gpu.global.u64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void st_release_u64(unsigned long long* p, unsigned long long v) {
  asm volatile("st.release.gpu.global.u64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

// Waits (bounded) until position j of the ready list carries this launch's
// epoch; returns the matrix published there, or -1.
__device__ int wait_ready_pos(const unsigned long long* list, int j, unsigned epoch,
                              const Ctx& c) {
  unsigned long long v = ld_acquire_u64(list + j);
  if (static_cast<unsigned>(v >> 32) == epoch) return static_cast<int>(static_cast<unsigned>(v));
  volatile int* ab = &c.B->abort;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    __nanosleep(128);
    v = ld_acquire_u64(list + j);
    if (static_cast<unsigned>(v >> 32) == epoch) return static_cast<int>(static_cast<unsigned>(v));
    if ((it & 63u) == 0) {
      if (*ab) return -1;
      if (ptx::globaltimer() - t0 > c.timeout_ns) {
        atomicOr(c.status, kDevTimeout);
        *ab = 1;
        return -1;
      }
    }
  }
}

struct Ring {
  int stage = 0;
  uint32_t phase = 0;
  __device__ __forceinline__ void next(int stages) {
    if (++stage == stages) {
      stage = 0;
      phase ^= 1u;
    }
  }
};


__device__ __forceinline__ float ld_elem(const void* base, int dtype, int64_t e) {
  return dtype == 0 ? static_cast<const float*>(base)[e]
                    : __bfloat162float(static_cast<const __nv_bfloat16*>(base)[e]);
}



// Block of C = A B owned by consumer thread t: rows TI (t / 16), columns
// TJ (t % 16) of LD x LD fp32 matrices in shared memory (row-major, leading
// dimension LD, entries outside m x m zero).  LD is 32 (m <= 32, 2 x 2
// blocks) or 64 (4 x 4 blocks), so the k loop is fully unrolled with no
// bounds; the k-sum runs in index order, so every CTA forms the same bits.
// C block = A B over k < K (K a multiple of 4, at most LD: the rows and
// columns past m are zero, so the sum may stop at m rounded up to 4).
// A block wholly outside the leading K x K (rows of A or columns of B past
// m, which are zero) is zero exactly and loads nothing: the products are
// bound by shared-memory wavefronts, so the threads of such blocks sit out.
template <int TI, int TJ, int LD>
__device__ __forceinline__ void mm_block(const float* A, const float* B, int i0, int j0,
                                         float (&acc)[TI][TJ], int K) {
#pragma unroll
  for (int r = 0; r < TI; ++r)
#pragma unroll
    for (int c = 0; c < TJ; ++c) acc[r][c] = 0.f;
  if (i0 >= K || j0 >= K) return;
#pragma unroll 2
  for (int k = 0; k < K; k += 4) {
    float a[TI][4], b[4][TJ];
#pragma unroll
    for (int r = 0; r < TI; ++r) {
      const float4 v = *reinterpret_cast<const float4*>(A + (i0 + r) * LD + k);
      a[r][0] = v.x; a[r][1] = v.y; a[r][2] = v.z; a[r][3] = v.w;
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk) {
      if constexpr (TJ == 4) {
        const float4 v = *reinterpret_cast<const float4*>(B + (k + kk) * LD + j0);
        b[kk][0] = v.x; b[kk][1] = v.y; b[kk][2] = v.z; b[kk][3] = v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(B + (k + kk) * LD + j0);
        b[kk][0] = v.x; b[kk][1] = v.y;
      }
    }
#pragma unroll
    for (int kk = 0; kk < 4; ++kk)
#pragma unroll
      for (int r = 0; r < TI; ++r)
#pragma unroll
        for (int c = 0; c < TJ; ++c) acc[r][c] = fmaf(a[r][kk], b[kk][c], acc[r][c]);
  }
}

template <int TI, int TJ, int LD>
__device__ __forceinline__ void st_block(float* C, int i0, int j0, const float (&v)[TI][TJ]) {
#pragma unroll
  for (int r = 0; r < TI; ++r) {
    if constexpr (TJ == 4)
      *reinterpret_cast<float4*>(C + (i0 + r) * LD + j0) = make_float4(v[r][0], v[r][1], v[r][2], v[r][3]);
    else
      *reinterpret_cast<float2*>(C + (i0 + r) * LD + j0) = make_float2(v[r][0], v[r][1]);
  }
}

__device__ __forceinline__ void cons_sync() { ptx::named_bar(kConsBar, kT); }

// Gram-space NS of one matrix, run by the consumers of the CTA whose item
// completed it: sums the partial Grams, normalises, iterates and writes
// Q / ||X0|| as the bf16 B-operand image (hi rows, then lo rows).  `gs`
// holds five LD x LD fp32 matrices (R, T, P, Q, Q') plus a few scalars.
// Per step three phases: {T = R^2, P = aI + bR + cT}, {T = P R, Q' = P Q},
// {R = T P} (the first step takes Q = P, the last needs neither R nor T).
template <int TI, int TJ, int LD, bool LOWMEM>
__device__ __noinline__ void gram_space(const SmallParams& p, int mat, float* gs, int t) {
  const int m = p.m;
  constexpr int MM = LD * LD;
  // Five LD x LD matrices: R, T = P R, P, Q and the next Q.  LOWMEM keeps
  // three (R also holds T between the two products of a step, Q is updated
  // in place): each product then goes through registers and a barrier, two
  // more barriers per step, which the latency-bound small Gram-space job
  // feels, so only the carve-ups that need the space use it.
  float* R = gs;
  float* P = gs + MM;
  float* Q = gs + 2 * MM;
  float* T = LOWMEM ? R : gs + 3 * MM;
  float* Qn = LOWMEM ? Q : gs + 4 * MM;
  float* sc = gs + (LOWMEM ? 3 : 5) * MM;
  // the 16 x 16 blocks of TI x TJ cover LD x LD: consumer threads 0..255
  // form the products, the others only take part in the barriers
  const bool blk = t < 256;
  const int K4 = (m + 3) & ~3;   // product length: m rounded up to 4
  const int i0 = TI * ((t & 255) >> 4), j0 = TJ * (t & 15);
  // R_0 (unnormalised) = sum of the item partials in block order.  The
  // m x m elements are dealt to the threads four at a time and the partial
  // loads of the four go out together, eight partials at a time (32 loads in
  // flight per thread: the sum is bound by L2 latency, not bandwidth).
  // Partial block q (item q / nblk, stacked block q % nblk) is at
  // part + (mat nb + q / nblk) pstride + (q % nblk) m^2.
  const float* part = p.part + static_cast<size_t>(mat) * p.nb * p.pstride;
  const int nblk = p.nblk;                 // 1 or 2: q / nblk and q % nblk as shift and mask
  const int bsh = nblk - 1;                // (a division by a run-time divisor here costs
  const int nq = p.nb * nblk;              // the job about 15 us at m = 24)
  const int mm = m * m;
  for (int e = t; e < MM; e += kT) R[e] = 0.f;   // padding rows and columns stay zero
  cons_sync();
  for (int base = 0; base < mm; base += 4 * kT) {
    int src[4];
    float acc[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      src[u] = base + u * kT + t;
      acc[u] = 0.f;
    }
    for (int b0 = 0; b0 < nq; b0 += 8) {
      float v[4][8];
#pragma unroll
      for (int b = 0; b < 8; ++b) {
        const int q = b0 + b;
        const float* pq = part + static_cast<size_t>(q >> bsh) * p.pstride + (q & bsh) * mm;
#pragma unroll
        for (int u = 0; u < 4; ++u) v[u][b] = (q < nq && src[u] < mm) ? __ldcg(pq + src[u]) : 0.f;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
#pragma unroll
        for (int b = 0; b < 8; ++b) acc[u] += v[u][b];
    }
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (src[u] < mm) {
        const int i = src[u] / m, j = src[u] - (src[u] / m) * m;
        R[i * LD + j] = acc[u];
      }
  }
  cons_sync();
  if (t < 32) {   // trace(X0 X0^T) = ||X0||_F^2, fp32, fixed reduction order
    float v = (t < m ? R[t * LD + t] : 0.f) + (t + 32 < m ? R[(t + 32) * LD + t + 32] : 0.f);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (t == 0) {
      if (!isfinite(v)) atomicOr(p.status, kDevNonfinite);
      sc[0] = 1.f / (sqrtf(v) + p.eps);
    }
  }
  cons_sync();
  const float inv = sc[0];
  const float s2 = inv * inv;
  for (int e = t; e < MM; e += kT) R[e] *= s2;
  cons_sync();
  for (int k = 0; k < p.steps; ++k) {
    const float a = p.coef[k][0], b = p.coef[k][1], c = p.coef[k][2];
    const bool more = k + 1 < p.steps;
    {   // T = R^2 (in registers), P = aI + bR + cR^2 (zero outside m x m)
      float acc[TI][TJ], pv[TI][TJ];
      if (blk) mm_block<TI, TJ, LD>(R, R, i0, j0, acc, K4);
#pragma unroll
      for (int r = 0; r < TI; ++r)
#pragma unroll
        for (int cc = 0; cc < TJ; ++cc) {
          const int i = i0 + r, j = j0 + cc;
          pv[r][cc] = (i < m && j < m)
                          ? fmaf(b, R[i * LD + j], c * acc[r][cc]) + (i == j ? a : 0.f)
                          : 0.f;
        }
      if (blk) st_block<TI, TJ, LD>(P, i0, j0, pv);
      if (blk && k == 0) st_block<TI, TJ, LD>(Q, i0, j0, pv);
    }
    cons_sync();
    if (more || k > 0) {
      if (LOWMEM) {
        // one product in registers at a time (the register budget of the
        // whole kernel follows its largest callee)
        float acc[TI][TJ];
        if (more) {
          if (blk) mm_block<TI, TJ, LD>(P, R, i0, j0, acc, K4);   // T = P R
          cons_sync();   // every thread has read R
          if (blk) st_block<TI, TJ, LD>(T, i0, j0, acc);
        }
        if (k > 0) {
          if (blk) mm_block<TI, TJ, LD>(P, Q, i0, j0, acc, K4);   // Q' = P Q
          cons_sync();   // every thread has read Q
          if (blk) st_block<TI, TJ, LD>(Qn, i0, j0, acc);
        }
      } else {
        float acc[TI][TJ];
        if (blk && more) {
          mm_block<TI, TJ, LD>(P, R, i0, j0, acc, K4);     // T = P R
          st_block<TI, TJ, LD>(T, i0, j0, acc);
        }
        if (blk && k > 0) {
          mm_block<TI, TJ, LD>(P, Q, i0, j0, acc, K4);     // Q' = P Q
          st_block<TI, TJ, LD>(Qn, i0, j0, acc);
        }
      }
      cons_sync();
      if (!LOWMEM && k > 0) {
        float* x = Q;
        Q = Qn;
        Qn = x;
      }
    }
    if (more) {
      float acc[TI][TJ];
      if (blk) mm_block<TI, TJ, LD>(T, P, i0, j0, acc, K4);          // R <- (P R) P
      if (LOWMEM) cons_sync();
      if (blk) st_block<TI, TJ, LD>(R, i0, j0, acc);
      cons_sync();
    }
  }
  if (p.steps == 0) {   // Q = I (the whole buffer: nothing else wrote it)
    for (int e = t; e < MM; e += kT) {
      const int i = e / LD;
      Q[e] = (i < m && e == i * LD + i) ? 1.f : 0.f;
    }
    cons_sync();
  }
  // Q / ||X0|| as bf16 hi (rows 0..nmm-1) then lo, K-major 128-byte-swizzled
  uint8_t* dst = p.qimg + static_cast<size_t>(mat) * p.qbytes;
  const int lo_off = p.nmm * 128;
  for (int cidx = t; cidx < p.nmm * 8; cidx += kT) {
    const int q = cidx >> 3, k0 = (cidx & 7) * 8;
    uint4 hi4, lo4;
    __nv_bfloat16* h = reinterpret_cast<__nv_bfloat16*>(&hi4);
    __nv_bfloat16* l = reinterpret_cast<__nv_bfloat16*>(&lo4);
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int kx = k0 + j;
      const float v = (q < m && kx < m) ? Q[q * LD + kx] * inv : 0.f;
      h[j] = __float2bfloat16_rn(v);
      l[j] = __float2bfloat16_rn(v - __bfloat162float(h[j]));
    }
    const uint32_t off = ptx::sw128_offset(q, (cidx & 7) * 16);
    __stcg(reinterpret_cast<uint4*>(dst + off), hi4);
    __stcg(reinterpret_cast<uint4*>(dst + lo_off + off), lo4);
  }
}

// ---- stage layout ---------------------------------------------------------------------
// A stage holds, for one range of X columns of one item:
//   first phase:  G tile (cw1 X columns) at byte 0, Mom tile at mom_off, and
//                 the X0 tile the consumers write (cw1 / 64 chunks) at x_off;
//   second phase: W tile (128 X columns) at byte 0 and the X0 tile (2 chunks,
//                 reloaded from the item's image) at x_off.
// A 2 KB zero gap follows the X0 tile: the apply's K padding (rows mr..nmm-1
// of the second chunk) reads it.  Row-major matrices give [m][cols] tiles,
// transposed ones [cols][m].  TMA fills out-of-matrix elements with zero.
// Results (M', the X0 image, W' or O) go from registers straight to global
// memory, so a stage is free once the consumers and the MMA issuer are done
// with it.
enum StageKind : int { kStageP1 = 0, kStageP2 = 1, kStageP1End = 2, kStageEnd = 3 };

// Stage descriptor flags
constexpr int kFirst = 1, kLast = 2;

__device__ __forceinline__ uint32_t mom_off(const SmallParams& p, const SmallSlice& S) {
  return static_cast<uint32_t>(p.m * p.cw1 * (S.g_dtype == 0 ? 4 : 2));
}

// Element-wise copy of a tile from global memory into a stage (slices whose
// rows are not TMA-legal), zero outside the matrix: `cols` X columns from gj0.
__device__ void copy_tile_in(const SmallParams& p, const SmallSlice& S, int dtype,
                             const void* gbase, int64_t moff, int64_t gj0, int cols, uint8_t* st,
                             int lane) {
  const int m = p.m, n = p.n;
  for (int idx = lane; idx < m * cols; idx += 32) {
    int r, c;
    if (!S.trans) {
      r = idx / cols;
      c = idx - r * cols;
    } else {
      c = idx / m;
      r = idx - c * m;
    }
    const uint32_t so = static_cast<uint32_t>(S.trans ? c * m + r : r * cols + c);
    const bool in = gj0 + c < n;
    const int64_t e = moff + (S.trans ? (gj0 + c) * m + r : static_cast<int64_t>(r) * n + gj0 + c);
    if (dtype == 0) reinterpret_cast<float*>(st)[so] = in ? static_cast<const float*>(gbase)[e] : 0.f;
    else
      reinterpret_cast<__nv_bfloat16*>(st)[so] =
          in ? static_cast<const __nv_bfloat16*>(gbase)[e] : __float2bfloat16_rn(0.f);
  }
}

// Per-item constants of the consumers, read once from the parameters (the
// per-stage code then touches no parameter memory).
struct ItemCfg {
  int m, mr, cw, nmm, n;
  int trans, gvec, wvec;   // transposed layout; 16-byte vector global access legal
  int esg, wdt;            // G element size; W dtype (0 f32, 1 bf16)
  int step;                // momentum step (else NS only)
  uint32_t mom_off, x_off;
  int chunk_bytes;
  float mu, decay, stepk;
  int nesterov;
  float* Mom;              // matrix base pointers (elements)
  void* W;
  int64_t col0;            // first X column of the item
  uint8_t* img;            // the item's X0 image
  const CUtensorMap* wmap; // the slice's W tile map (TMA-legal W only)
  int z;                   // matrix index within the slice
  int tma_store;           // second phase: W' leaves through the stage by one TMA store
};

__device__ __forceinline__ ItemCfg item_cfg(const SmallParams& p, int item) {
  const int mat = item / p.nb;
  int si = 0;
  while (si + 1 < p.n_slices && mat >= p.s[si + 1].mat_base) ++si;
  const SmallSlice& S = p.s[si];
  const int64_t moff = static_cast<int64_t>(mat - S.mat_base) * p.m * p.n;
  ItemCfg c;
  c.m = p.m;
  c.mr = p.mr;
  c.cw = p.cw1;
  c.nmm = p.nmm;
  c.n = p.n;
  c.trans = S.trans;
  c.gvec = S.gbulk;
  c.wvec = S.wbulk;
  c.esg = S.g_dtype == 0 ? 4 : 2;
  c.wdt = S.w_dtype;
  c.step = p.step_mode;
  c.mom_off = static_cast<uint32_t>(p.m * p.cw1 * c.esg);
  c.x_off = static_cast<uint32_t>(p.x_off);
  c.chunk_bytes = p.mr * 128;
  c.mu = p.mu;
  c.decay = 1.f - p.lr * p.wd;
  c.stepk = p.lr * S.scale;
  c.nesterov = p.nesterov;
  c.Mom = S.Mom ? S.Mom + moff : nullptr;
  c.W = static_cast<uint8_t*>(S.W) + moff * (S.w_dtype == 0 ? 4 : 2);
  c.col0 = static_cast<int64_t>(item - mat * p.nb) * p.wb;
  c.img = p.ximg + static_cast<size_t>(item) * p.xbytes;
  c.wmap = &p.tm[si][2];
  c.z = mat - S.mat_base;
  c.tma_store = p.p2_tma_store && S.wbulk && !S.trans;
  return c;
}

// ---- consumers: first-phase stage ----------------------------------------------------
template <int ESG>
__device__ __forceinline__ void load8_smem(const uint8_t* base, int so, float* v) {
  if constexpr (ESG == 2) {
    const uint4 u = *reinterpret_cast<const uint4*>(base + so * 2);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const float2 f = __bfloat1622float2(h[j]);
      v[2 * j] = f.x;
      v[2 * j + 1] = f.y;
    }
  } else {
    const float4 a = *reinterpret_cast<const float4*>(base + so * 4);
    const float4 b = *reinterpret_cast<const float4*>(base + so * 4 + 16);
    v[0] = a.x; v[1] = a.y; v[2] = a.z; v[3] = a.w;
    v[4] = b.x; v[5] = b.y; v[6] = b.z; v[7] = b.w;
  }
}

// Momentum for 8 elements; d = the NS input (Nesterov or plain momentum).
template <bool STEP>
__device__ __forceinline__ void momentum8(const ItemCfg& c, const float* gv, float* mo, float* d) {
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if constexpr (STEP) {
      mo[j] = fmaf(c.mu, mo[j], gv[j]);                       // M_t = mu M_{t-1} + G
      d[j] = c.nesterov ? fmaf(c.mu, mo[j], gv[j]) : mo[j];
    } else {
      d[j] = gv[j];
    }
  }
}

// 8 contiguous M' values to global memory (nv of them inside the matrix).
__device__ __forceinline__ void store_mom8(float* dst, int nv, bool vec, const float* v) {
  if (vec && nv == 8) {
    __stcs(reinterpret_cast<float4*>(dst), make_float4(v[0], v[1], v[2], v[3]));
    __stcs(reinterpret_cast<float4*>(dst + 4), make_float4(v[4], v[5], v[6], v[7]));
  } else {
#pragma unroll
    for (int j = 0; j < 8; ++j)
      if (j < nv) dst[j] = v[j];
  }
}

// First-phase stage of X columns [c0, c0 + cw1) of the item: M' to global
// memory, X0 = bf16(D) into the stage's X0 tile (rows mr, cw1 / 64 chunks;
// rows m..mr-1 and columns outside the matrix zero) and to the item's image.
template <int ESG, bool STEP, bool PRECISE>
__device__ void consume_p1(const ItemCfg& c, int c0, uint8_t* st, int t) {
  const int m = c.m, cw = c.cw, cb = c.chunk_bytes;
  const uint8_t* smom = st + c.mom_off;
  uint8_t* sx = st + c.x_off;
  const int64_t gjs = c.col0 + c0;             // first global X column of the stage
  const int ncols = static_cast<int>(min(static_cast<int64_t>(cw), c.n - gjs));
  if (!c.trans) {
    // mr * cw1 / 8 <= 512 groups of 8: at most two per thread, whose shared
    // loads are all issued first
    const int gpr = cw >> 3;
    const int sh = gpr == 16 ? 4 : 3;                  // cw1 is 128 or 64
    const int ng = c.mr * gpr;
    float gv[2][8], mo[2][8];
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int g = t + u * kT;
      const int r = g >> sh;
      if (g < ng && r < m) {
        const int so = r * cw + ((g & (gpr - 1)) << 3);
        load8_smem<ESG>(st, so, gv[u]);
        if constexpr (STEP) load8_smem<4>(smom, so, mo[u]);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) gv[u][j] = mo[u][j] = 0.f;
      }
    }
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      const int g = t + u * kT;
      if (g >= ng) continue;
      const int r = g >> sh, c8 = (g & (gpr - 1)) << 3;
      float d[8];
      momentum8<STEP>(c, gv[u], mo[u], d);
      if constexpr (STEP) {
        if (r < m && c8 < ncols)
          store_mom8(c.Mom + static_cast<int64_t>(r) * c.n + gjs + c8, min(8, ncols - c8), c.gvec, mo[u]);
      }
      uint4 q;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
      for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(d[2 * j], d[2 * j + 1]);
      const uint32_t off = ptx::sw128_offset(r, (c8 & 63) * 2);
      constexpr int xs = PRECISE ? 2 : 1;   // chunk regions per 64 columns
      *reinterpret_cast<uint4*>(sx + (c8 >> 6) * xs * cb + off) = q;
      __stcg(reinterpret_cast<uint4*>(c.img + ((c0 + c8) >> 6) * xs * cb + off), q);
      if constexpr (PRECISE) {
        // lo = bf16(d - hi): X0 = hi + lo to about 16 significant bits
        uint4 ql;
        __nv_bfloat162* l = reinterpret_cast<__nv_bfloat162*>(&ql);
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const float2 hf = __bfloat1622float2(h[j]);
          l[j] = __floats2bfloat162_rn(d[2 * j] - hf.x, d[2 * j + 1] - hf.y);
        }
        *reinterpret_cast<uint4*>(sx + ((c8 >> 6) * 2 + 1) * cb + off) = ql;
        __stcg(reinterpret_cast<uint4*>(c.img + (((c0 + c8) >> 6) * 2 + 1) * cb + off), ql);
      }
    }
  } else {
    const int ig = c.mr >> 3;
    const float inv_ig = 1.f / static_cast<float>(ig);
    for (int g = t; g < cw * ig; g += kT) {
      const int cc = __float2int_rd((static_cast<float>(g) + 0.5f) * inv_ig);
      const int r = (g - cc * ig) << 3;
      const int nv = min(8, m - r);
      const int so = cc * m + r;
      float gv[8], mo[8], d[8];
      if (nv == 8 && c.gvec) {
        load8_smem<ESG>(st, so, gv);
        if constexpr (STEP) load8_smem<4>(smom, so, mo);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          gv[j] = j < nv ? ld_elem(st, ESG == 4 ? 0 : 1, so + j) : 0.f;
          mo[j] = (STEP && j < nv) ? reinterpret_cast<const float*>(smom)[so + j] : 0.f;
        }
      }
      momentum8<STEP>(c, gv, mo, d);
      if constexpr (STEP) {
        if (cc < ncols && nv > 0) store_mom8(c.Mom + (gjs + cc) * m + r, nv, c.gvec != 0, mo);
      }
      const int ci = c0 + cc;
      const uint32_t byte = (cc & 63) * 2, ibyte = (ci & 63) * 2;
      constexpr int xs = PRECISE ? 2 : 1;   // chunk regions per 64 columns
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const float dv = j < nv ? d[j] : 0.f;
        const __nv_bfloat16 v = __float2bfloat16_rn(dv);
        *reinterpret_cast<__nv_bfloat16*>(sx + (cc >> 6) * xs * cb + ptx::sw128_offset(r + j, byte)) = v;
        *reinterpret_cast<__nv_bfloat16*>(c.img + (ci >> 6) * xs * cb + ptx::sw128_offset(r + j, ibyte)) = v;
        if constexpr (PRECISE) {
          const __nv_bfloat16 lv = __float2bfloat16_rn(dv - __bfloat162float(v));
          *reinterpret_cast<__nv_bfloat16*>(sx + ((cc >> 6) * 2 + 1) * cb + ptx::sw128_offset(r + j, byte)) = lv;
          *reinterpret_cast<__nv_bfloat16*>(c.img + ((ci >> 6) * 2 + 1) * cb + ptx::sw128_offset(r + j, ibyte)) = lv;
        }
      }
    }
  }
}

template <bool PRECISE>
__device__ void consume_p1_dt(const ItemCfg& c, int c0, uint8_t* st, int t) {
  if (c.esg == 4) {
    if (c.step) consume_p1<4, true, PRECISE>(c, c0, st, t);
    else consume_p1<4, false, PRECISE>(c, c0, st, t);
  } else {
    if (c.step) consume_p1<2, true, PRECISE>(c, c0, st, t);
    else consume_p1<2, false, PRECISE>(c, c0, st, t);
  }
}



// ---- consumers: second-phase stage -------------------------------------------------------
template <typename WT>
__device__ __forceinline__ float w_ld(const WT* p, int i) {
  if constexpr (sizeof(WT) == 4) return p[i];
  else return __bfloat162float(p[i]);
}

template <typename WT>
__device__ __forceinline__ void w_st(WT* p, int64_t i, float v) {
  if constexpr (sizeof(WT) == 4) __stcs(p + i, v);
  else p[i] = __float2bfloat16_rn(v);
}

// 128-column tile at item column c0: O = D[:, q] + D[:, nmm + q] (X0 Q_hi^T +
// X0 Q_lo^T) from the TMEM slot, W' = decay W - stepk O (W from the stage) or
// O, to global memory.  The tile belongs to one set of four warps (the sets
// take alternate stages); warp q4 of the set owns lanes 32 q4.. (the
// columns) and every row.  Row-major tiles are written back into the stage first and
// leave as 4-column vectors (one 128-bit store per lane and 4 rows per warp
// instruction instead of one scalar store per element).
template <typename WT, bool STEP>
__device__ __forceinline__ void epi_tile(const ItemCfg& c, int c0, uint8_t* st, uint32_t oslot,
                                         int set, int q4, int lane, float* scr, uint64_t* stw,
                                         const Ctx& ctx) {
  const int m = c.m, nmm = c.nmm;
  const float decay = c.decay, stepk = c.stepk;
  WT* ws = reinterpret_cast<WT*>(st);
  const int col = 32 * q4 + lane;
  const int64_t gj = c.col0 + c0 + col;
  const uint32_t lq = static_cast<uint32_t>(32 * q4) << 16;
  WT* wg = static_cast<WT*>(c.W);
  if (c.tma_store) {
    // W' (or O) in place of W in the stage's [m][128] tile, then one TMA
    // store of the tile (columns and rows outside the matrix are clipped);
    // the set's leader waits until the store has read the stage before its
    // warp hands the stage back
    for (int q0 = 0; q0 < m; q0 += 4) {
      uint32_t rh[4], rl[4];
      ptx::tmem_ld_32x32b_x4(oslot + q0 + lq, rh);
      ptx::tmem_ld_32x32b_x4(oslot + nmm + q0 + lq, rl);
      float w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = (STEP && q0 + j < m) ? w_ld(ws, (q0 + j) * 128 + col) : 0.f;
      ptx::tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if (q0 + j < m) {
          const float o = __uint_as_float(rh[j]) + __uint_as_float(rl[j]);
          const float v = STEP ? fmaf(decay, w[j], -stepk * o) : o;
          if constexpr (sizeof(WT) == 4) ws[(q0 + j) * 128 + col] = v;
          else ws[(q0 + j) * 128 + col] = __float2bfloat16_rn(v);
        }
      }
    }
    // every writer's stores are made visible to the TMA (async proxy), each
    // warp arrives on the stage's barrier, and the leader waits for the
    // phase its own arrival names (bounded: a warp that gave up costs a
    // timeout, never a hang; the stage is not reused before the leader's
    // warp hands it back, so no arrival of a later use can complete it)
    ptx::fence_proxy_async_smem();
    __syncwarp();
    if (lane == 0) {
      if (q4 == 0) {
        const uint64_t tok = ptx::mbar_arrive_token(stw);
        if (mwait_token(stw, tok, ctx) && dbg_ok(((c.col0 + c0) & 7) == 0, ctx.status)) {
          ptx::tma_store_3d(c.wmap, ws, static_cast<int>(c.col0 + c0), 0, c.z);
          ptx::bulk_commit();
          ptx::bulk_wait_read<0>();
        }
      } else {
        ptx::mbar_arrive(stw);
      }
    }
    return;
  }
  if (!c.trans) {
    const int64_t gjw = c.col0 + c0 + 32 * q4;    // first global column of this warp
    const bool vec = c.wvec && sizeof(WT) == 4 && gjw + 32 <= c.n;
    for (int q0 = 0; q0 < m; q0 += 4) {
      uint32_t rh[4], rl[4];
      ptx::tmem_ld_32x32b_x4(oslot + q0 + lq, rh);
      ptx::tmem_ld_32x32b_x4(oslot + nmm + q0 + lq, rl);
      float w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) w[j] = (STEP && q0 + j < m) ? w_ld(ws, (q0 + j) * 128 + col) : 0.f;
      ptx::tmem_ld_wait();
      float v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float o = __uint_as_float(rh[j]) + __uint_as_float(rl[j]);
        v[j] = STEP ? fmaf(decay, w[j], -stepk * o) : o;
      }
      if (vec) {
        // rows q0..q0+3 x the warp's 32 columns through the warp's scratch
        // (not the stage, which TMA refills), then lane l stores row
        // q0 + l / 8, columns 4 (l % 8) .. + 3 of the warp
#pragma unroll
        for (int j = 0; j < 4; ++j) scr[j * 32 + lane] = v[j];
        __syncwarp();
        const int rr = lane >> 3, cc = 4 * (lane & 7);
        if (q0 + rr < m) {
          const float4 x = *reinterpret_cast<const float4*>(scr + rr * 32 + cc);
          __stcs(reinterpret_cast<float4*>(reinterpret_cast<float*>(wg) + static_cast<int64_t>(q0 + rr) * c.n +
                                           c.col0 + c0 + 32 * q4 + cc), x);
        }
        __syncwarp();
      } else if (gj < c.n) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if (q0 + j < m) w_st(wg, static_cast<int64_t>(q0 + j) * c.n + gj, v[j]);
      }
    }
  } else {
    const bool live = gj < c.n;
    WT* wrow = wg + gj * m;
    for (int cq = 0; cq < nmm; cq += 16) {
      uint32_t rh[16], rl[16];
      ptx::tmem_ld_32x32b_x16(oslot + cq + lq, rh);
      ptx::tmem_ld_32x32b_x16(oslot + nmm + cq + lq, rl);
      float w[16];
#pragma unroll
      for (int j = 0; j < 16; ++j) w[j] = (STEP && cq + j < m) ? w_ld(ws, col * m + cq + j) : 0.f;
      ptx::tmem_ld_wait();
      if (!live) continue;
#pragma unroll
      for (int j = 0; j < 16; ++j) {
        if (cq + j < m) {
          const float o = __uint_as_float(rh[j]) + __uint_as_float(rl[j]);
          w_st(wrow, cq + j, STEP ? fmaf(decay, w[j], -stepk * o) : o);
        }
      }
    }
  }
}

__device__ void epi_tile_any(const ItemCfg& c, int c0, uint8_t* st, uint32_t oslot, int set,
                             int q4, int lane, float* scr, uint64_t* stw, const Ctx& ctx) {
  if (c.wdt == 0) {
    if (c.step) epi_tile<float, true>(c, c0, st, oslot, set, q4, lane, scr, stw, ctx);
    else epi_tile<float, false>(c, c0, st, oslot, set, q4, lane, scr, stw, ctx);
  } else {
    if (c.step) epi_tile<__nv_bfloat16, true>(c, c0, st, oslot, set, q4, lane, scr, stw, ctx);
    else epi_tile<__nv_bfloat16, false>(c, c0, st, oslot, set, q4, lane, scr, stw, ctx);
  }
}

struct ItemRef {
  int si;          // slice
  int mat;         // matrix within the launch
  int64_t moff;    // element offset of the matrix
  int64_t col0;    // first X column of the item
};

__device__ __forceinline__ ItemRef item_ref(const SmallParams& p, int item) {
  ItemRef r;
  r.mat = item / p.nb;
  r.si = 0;
  while (r.si + 1 < p.n_slices && r.mat >= p.s[r.si + 1].mat_base) ++r.si;
  r.moff = static_cast<int64_t>(r.mat - p.s[r.si].mat_base) * p.m * p.n;
  r.col0 = static_cast<int64_t>(item - r.mat * p.nb) * p.wb;
  return r;
}

}  // namespace

// PRECISE: X0 carried as bf16 hi + lo (its own instantiation, so that the
// common path carries none of it).
template <bool PRECISE>
__global__ void __launch_bounds__(kSmallThreads, 1)
    ns_small_kernel(const __grid_constant__ SmallParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* ring = sm + p.off_ring;          // stage s at ring + s * stage_bytes
  float* gs = reinterpret_cast<float*>(sm + p.off_gs);
  SmallBars* B = reinterpret_cast<SmallBars*>(sm + p.off_bar);
  const Ctx ctx{B, p.status, p.timeout_ns};
  // This launch's counters (ready-list length, claimed second- and first-
  // phase items) are slot epoch % 64 of a ring, its per-matrix arrivals slot
  // epoch % 2 of two; the previous launch zeroed both, CTA 0 zeroes the next
  // launch's.
  unsigned* lctr = p.ctr + (p.epoch % kSmallCtrSlots) * 4;
  unsigned* larr = p.arrive + static_cast<size_t>(p.epoch & 1u) * p.cap;
  if (blockIdx.x == 0) {
    if (threadIdx.x < 4) p.ctr[((p.epoch + 1) % kSmallCtrSlots) * 4 + threadIdx.x] = 0u;
    unsigned* nxt = p.arrive + static_cast<size_t>((p.epoch + 1) & 1u) * p.cap;
    for (int i = threadIdx.x; i < p.cap; i += kSmallThreads) nxt[i] = 0u;
  }

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int m = p.m, nmm = p.nmm, wb = p.wb, NS = p.stages;
  const int chunk_bytes = p.mr * 128;
  const int tiles = wb / 128;
  const int s1 = wb / p.cw1;               // first-phase stages per item
  const int oslot_cols = 2 * ((nmm + 31) & ~31);   // O slot: X0 Q_hi^T then X0 Q_lo^T
  // First-phase Gram MMA: the stage's two 64-column chunks stacked as one
  // 2 mr-row operand (m <= 32), or, precise, each chunk's [hi; lo] stacked
  // (the four blocks hi hi^T, hi lo^T, lo hi^T, lo lo^T sum to X0 X0^T).
  const bool stack = p.cw1 == 128 || PRECISE;
  const int ngram = stack ? 2 * p.mr : nmm;          // Gram MMA N
  constexpr int xs = PRECISE ? 2 : 1;                // chunk regions per 64 X0 columns
  const uint32_t obase = 2 * p.gcols;                // first O slot column

  if (tid == 0) {
    for (int i = 0; i < kSmallMaxStages; ++i) {
      ptx::mbar_init(&B->ring_full[i], 1);
      ptx::mbar_init(&B->cons_done[i], kT / 32);
      ptx::mbar_init(&B->mma_done[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&B->gram_full[i], 1);
      ptx::mbar_init(&B->q_full[i], 1);
      ptx::mbar_init(&B->q_free[i], 1);
    }
    ptx::mbar_init(&B->mma_fin, 1);
    for (int i = 0; i < kSmallMaxStages; ++i) ptx::mbar_init(&B->st_w[i], 4);
    B->last = 0;
    B->abort = 0;
    ptx::fence_mbar_init();
  }
  // zero gap after every stage's X0 tile (read as the apply's K padding)
  for (int s = 0; s < NS; ++s)
    for (int i = tid; i < 2048 / 16; i += kSmallThreads)
      reinterpret_cast<uint4*>(ring + s * p.stage_bytes + p.x_off + 2 * xs * chunk_bytes)[i] =
          make_uint4(0, 0, 0, 0);
  if (warp == 1) ptx::tmem_alloc(&B->tslot, kSmallTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = B->tslot;

  if (warp == 0) {
    // ======================= producer (loads) =======================
    // the descriptors of the tensor maps this launch uses, fetched ahead of
    // the first loads
    if (lane < p.n_slices) {
      const SmallSlice& S = p.s[lane];
      if (S.gbulk) {
        ptx::prefetch_tmap(&p.tm[lane][0]);
        if (p.step_mode) ptx::prefetch_tmap(&p.tm[lane][1]);
      }
      if (p.step_mode && S.wbulk) ptx::prefetch_tmap(&p.tm[lane][2]);
    }
    // Launch constants in registers, and per item (first phase) or per claim
    // (second phase) one load plan: reading the parameter block's slice
    // fields on every stage cost the producer about 0.2 us per stage, and
    // in the second phase the producer sets the pace.
    const int stage_bytes = p.stage_bytes, cw1 = p.cw1, x_off = p.x_off;
    const int xbytes = p.xbytes, nb = p.nb, n_items = p.items, total_mats = p.total_mats;
    const int qbytes = p.qbytes, off_q = p.off_q;
    const bool step_mode = p.step_mode != 0;
    uint8_t* const ximg = p.ximg;
    const uint8_t* const qimg = p.qimg;
    const unsigned long long* const ready_list = p.ready_list;
    const unsigned epoch = p.epoch;
    struct LoadPlan {
      int item = -1;
      int z = 0, trans = 0;        // matrix within its slice; stored transposed
      int64_t col0 = 0;            // first X column of the item
      bool bulk = false;           // the data tile(s) by TMA (else element-wise)
      uint32_t tx = 0;             // bytes the stage's asynchronous copies deliver
      uint32_t mom_off = 0;        // Mom tile inside the stage (first phase)
      const CUtensorMap* tm = nullptr;   // G (then Mom) map, or the W map
      const uint8_t* img = nullptr;      // the item's X0 image (second phase)
    };
    auto make_plan = [&](int kind, int item) {
      LoadPlan L;
      L.item = item;
      const ItemRef ir = item_ref(p, item);
      const SmallSlice& S = p.s[ir.si];
      L.z = ir.mat - S.mat_base;
      L.trans = S.trans;
      L.col0 = ir.col0;
      if (kind == kStageP1) {
        L.bulk = S.gbulk != 0;
        L.tm = &p.tm[ir.si][0];
        L.mom_off = mom_off(p, S);
        if (L.bulk) L.tx = static_cast<uint32_t>(m * cw1 * ((S.g_dtype == 0 ? 4 : 2) + (step_mode ? 4 : 0)));
      } else {
        L.bulk = step_mode && S.wbulk;
        L.tm = &p.tm[ir.si][2];
        L.img = ximg + static_cast<size_t>(item) * xbytes;
        L.tx = static_cast<uint32_t>(2 * xs * chunk_bytes);
        if (L.bulk) L.tx += static_cast<uint32_t>(m * 128 * (S.w_dtype == 0 ? 4 : 2));
      }
      return L;
    };
    Ring rg;
    bool ok = true;
    int nput = 0;                 // stages handed out (stage j % NS, parity (j / NS) & 1)
    int qk_last[2] = {-1, -1};    // lane 0: last claim whose Q image went to buffer b
    // Hands the next stage to the other roles once its previous use is done
    // (consumers and MMA issuer): descriptor, then the tile(s).  Element-wise
    // copies (slices whose rows are not TMA-legal) go through the slice.
    auto put = [&](int kind, const LoadPlan& L, int c0, int flags) -> bool {
      if (!mwait_warp(&B->cons_done[rg.stage], rg.phase ^ 1u, ctx)) return false;
      if (!mwait_warp(&B->mma_done[rg.stage], rg.phase ^ 1u, ctx)) return false;
      uint8_t* st = ring + rg.stage * stage_bytes;
      uint64_t* full = &B->ring_full[rg.stage];
      const bool data = kind == kStageP1 || kind == kStageP2;
      if (data && !L.bulk && (kind == kStageP1 || step_mode)) {
        const ItemRef ir = item_ref(p, L.item);
        const SmallSlice& S = p.s[ir.si];
        const int64_t gj0 = ir.col0 + c0;
        if (kind == kStageP1) {
          copy_tile_in(p, S, S.g_dtype, S.G, ir.moff, gj0, cw1, st, lane);
          if (step_mode) copy_tile_in(p, S, 0, S.Mom, ir.moff, gj0, cw1, st + L.mom_off, lane);
        } else {
          copy_tile_in(p, S, S.w_dtype, S.W, ir.moff, gj0, 128, st, lane);
        }
      }
      __syncwarp();
      if (lane == 0) {
        B->desc[rg.stage][0] = kind;
        B->desc[rg.stage][1] = data ? L.item : -1;
        B->desc[rg.stage][2] = c0;
        B->desc[rg.stage][3] = flags;
        if (data && L.tx) {
          // TMA coordinates of the tile at X column gj0 (X columns are the
          // stored rows of a transposed matrix)
          const int64_t gj0 = L.col0 + c0;
          const int x = L.trans ? 0 : static_cast<int>(gj0);
          const int y = L.trans ? static_cast<int>(gj0) : 0;
          ptx::mbar_arrive_expect_tx(full, L.tx);
          // debug builds: the innermost coordinate is a multiple of 16 bytes
          // for both the bf16 and the fp32 tensor; the image copy is aligned
          const uint8_t* img = L.img + (c0 / 64) * xs * chunk_bytes;
          const uint32_t img_bytes = static_cast<uint32_t>(2 * xs * chunk_bytes);
          if (!dbg_ok((x & 7) == 0, ctx.status)) {
          } else if (kind == kStageP1) {
            ptx::tma_load_3d(st, L.tm, full, x, y, L.z);
            if (step_mode) ptx::tma_load_3d(st + L.mom_off, L.tm + 1, full, x, y, L.z);
          } else if (dbg_ok(((reinterpret_cast<uintptr_t>(img) | img_bytes |
                              ptx::smem_u32(st + x_off)) & 15) == 0,
                            ctx.status)) {
            if (L.bulk) ptx::tma_load_3d(st, L.tm, full, x, y, L.z);
            ptx::bulk_load(st + x_off, img, img_bytes, full);
          }
        } else {
          ptx::mbar_arrive(full);
        }
      }
      __syncwarp();
      rg.next(NS);
      ++nput;
      return true;
    };
    const LoadPlan none;
    // First phase: items are claimed in increasing order from a launch-wide
    // counter, so a CTA that spends time on a Gram-space step simply takes
    // fewer items.
    for (;;) {
      int item = -1;
      if (lane == 0) {
        const unsigned c = atomicAdd(lctr + 2, 1u);
        if (c < static_cast<unsigned>(n_items)) item = static_cast<int>(c);
      }
      item = __shfl_sync(0xffffffffu, item, 0);
      if (item < 0) break;
      const LoadPlan L = make_plan(kStageP1, item);
      for (int s = 0; s < s1 && ok; ++s)
        ok = put(kStageP1, L, s * cw1, (s == 0 ? kFirst : 0) | (s == s1 - 1 ? kLast : 0));
      if (!ok) break;
    }
    if (ok) ok = put(kStageP1End, none, 0, 0);
    // Second phase: work is claimed in the order matrices were published
    // (position j of the ready list, item, unit of the item), so no CTA
    // waits for a late matrix while published work remains.  The unit is
    // p2_tiles tiles; a claim takes up to p2_units consecutive units, fewer
    // as the work runs out (guided self-scheduling: the remaining units over
    // twice the CTA count), so the claims' atomics and ready-list reads are
    // paid once per several units while the launch ends on small claims.
    // A claim is walked as segments (its units within one item), each with
    // its own Q image (buffer k & 1 for segment k).
    const int tpu = p.p2_tiles;                       // tiles per unit
    const int parts = (tiles + tpu - 1) / tpu;        // units per item
    const unsigned per = static_cast<unsigned>(nb * parts);
    const unsigned total_units = per * static_cast<unsigned>(total_mats);
    const unsigned max_take = static_cast<unsigned>(p.p2_units);
    const unsigned ctas2 = 2u * gridDim.x;
    unsigned take = max_take;
    int k = 0;
    while (ok) {
      unsigned start = 0;
      if (lane == 0) start = atomicAdd(lctr + 1, take);
      start = __shfl_sync(0xffffffffu, start, 0);
      if (start >= total_units) break;
      const unsigned end = min(start + take, total_units);
      const unsigned left = total_units - end;
      take = max(1u, min(max_take, left / ctas2));
      for (unsigned u = start; u < end && ok; ++k) {
        const int j = static_cast<int>(u / per);
        const unsigned rem = u - static_cast<unsigned>(j) * per;
        const int it_m = static_cast<int>(rem / parts);                // item within the matrix
        const unsigned item_end = static_cast<unsigned>(j) * per + (it_m + 1) * parts;
        const unsigned seg_end = min(end, item_end);
        const int t0 = static_cast<int>(rem % parts) * tpu;
        const int t1 = min(tiles, t0 + static_cast<int>(seg_end - u) * tpu);
        const int b = k & 1;
        int item = -1;
        if (lane == 0) {
          const int mat = wait_ready_pos(ready_list, j, epoch, ctx);
          if (mat >= 0) item = mat * nb + it_m;
          // Q buffer b is free once the MMAs of segment k-2 are done
          if (item >= 0 && !mwait(&B->q_free[b], ((k >> 1) & 1) ^ 1u, ctx)) item = -1;
          if (item >= 0) {
            ptx::fence_proxy_async_global();
            ptx::mbar_arrive_expect_tx(&B->q_full[b], static_cast<uint32_t>(qbytes));
            const uint8_t* qsrc = qimg + static_cast<size_t>(item / nb) * qbytes;
            if (dbg_ok(((reinterpret_cast<uintptr_t>(qsrc) | static_cast<uintptr_t>(qbytes)) & 15) == 0,
                       ctx.status))
              ptx::bulk_load(sm + off_q + b * qbytes, qsrc, static_cast<uint32_t>(qbytes),
                             &B->q_full[b]);
            qk_last[b] = k;
          }
        }
        item = __shfl_sync(0xffffffffu, item, 0);
        if (item < 0) {
          ok = false;
          break;
        }
        const LoadPlan L = make_plan(kStageP2, item);
        for (int t = t0; t < t1 && ok; ++t)
          ok = put(kStageP2, L, 128 * t, (t == t0 ? kFirst : 0) | (t == t1 - 1 ? kLast : 0));
        u = seg_end;
      }
    }
    put(kStageEnd, none, 0, 0);
    // No copy may still target this CTA's shared memory at exit, also after
    // an abort: the last (up to) NS stages handed out and the last Q image
    // of each buffer have landed.
    if (lane == 0) {
      for (int j = nput > NS ? nput - NS : 0; j < nput; ++j)
        mwait_drain(&B->ring_full[j % NS], static_cast<uint32_t>(j / NS) & 1u, ctx);
      for (int b = 0; b < 2; ++b)
        if (qk_last[b] >= 0) mwait_drain(&B->q_full[b], static_cast<uint32_t>(qk_last[b] >> 1) & 1u, ctx);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ======================= MMA issuer =======================
    const uint32_t idesc_gram = ptx::idesc_bf16_f32(128, ngram);
    const uint32_t idesc_app = ptx::idesc_bf16_f32(128, 2 * nmm) | (1u << 15);   // A MN-major
    if (lane == 0) {
      Ring rg;
      int k1 = 0, k2 = -1;
      for (;;) {
        if (!mwait(&B->ring_full[rg.stage], rg.phase, ctx)) break;
        const int kind = B->desc[rg.stage][0];
        const int flags = B->desc[rg.stage][3];
        if (kind == kStageEnd) break;
        const uint32_t sx = ptx::smem_u32(ring + rg.stage * p.stage_bytes + p.x_off);
        if (kind == kStageP1) {
          // partial Gram of this stage's X0 tile into accumulator k1 & 1: the
          // two 64-column chunks stacked as 2 mr rows (or one chunk), 4 K-steps
          if (!mwait(&B->cons_done[rg.stage], rg.phase, ctx)) break;
          ptx::tc_fence_after();
          const int g = k1 & 1;
          if (PRECISE) {
            // each 64-column chunk's [hi; lo] is one operand
            for (int ch = 0; ch < p.cw1 / 64; ++ch)
#pragma unroll
              for (int kk = 0; kk < 4; ++kk) {
                const uint64_t d = ptx::sdesc_kmajor_sw128(sx + ch * 2 * chunk_bytes + kk * 32);
                ptx::umma_bf16(tmem + p.gcols * g, d, d, idesc_gram,
                               ((flags & kFirst) && ch == 0 && kk == 0) ? 0u : 1u);
              }
          } else {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              const uint64_t d = ptx::sdesc_kmajor_sw128(sx + kk * 32);
              ptx::umma_bf16(tmem + 64 * g, d, d, idesc_gram, ((flags & kFirst) && kk == 0) ? 0u : 1u);
            }
          }
          ptx::umma_commit(&B->mma_done[rg.stage]);
          if (flags & kLast) {
            ptx::umma_commit(&B->gram_full[g]);
            ++k1;
          }
        } else if (kind == kStageP2) {
          if (flags & kFirst) {
            ++k2;
            if (!mwait(&B->q_full[k2 & 1], (k2 >> 1) & 1, ctx)) break;
          }
          ptx::tc_fence_after();
          // X0 (MN-major, 128 columns) times [Q_hi; Q_lo]^T: one MMA per K-step
          const uint32_t sq = ptx::smem_u32(sm + p.off_q + (k2 & 1) * p.qbytes);
          const uint32_t ocol = obase + oslot_cols * rg.stage;
          if (PRECISE) {
            // the hi chunks, then the lo chunks one region later
            for (int j = 0; j < nmm / 16; ++j) {
              const uint64_t b = ptx::sdesc_kmajor_sw128(sq + j * 32);
              for (int hl = 0; hl < 2; ++hl) {
                const uint64_t a =
                    ptx::sdesc_mnmajor_sw128(sx + hl * chunk_bytes + j * 2048, 2 * chunk_bytes, 1024);
                ptx::umma_bf16(tmem + ocol, a, b, idesc_app, (j != 0 || hl != 0) ? 1u : 0u);
              }
            }
          } else {
            for (int j = 0; j < nmm / 16; ++j) {
              const uint64_t a = ptx::sdesc_mnmajor_sw128(sx + j * 2048, chunk_bytes, 1024);
              ptx::umma_bf16(tmem + ocol, a, ptx::sdesc_kmajor_sw128(sq + j * 32), idesc_app,
                             j != 0 ? 1u : 0u);
            }
          }
          ptx::umma_commit(&B->mma_done[rg.stage]);
          if (flags & kLast) ptx::umma_commit(&B->q_free[k2 & 1]);
        } else {
          // keep mma_done[s] at one completion per use of the stage
          ptx::mbar_arrive(&B->mma_done[rg.stage]);
        }
        rg.next(NS);
      }
      // no MMA may still run when TMEM is freed (after an abort nobody
      // waits for the last ones)
      ptx::umma_commit(&B->mma_fin);
      mwait_drain(&B->mma_fin, 0, ctx);
    }
    __syncwarp();
  } else {
    // ======================= consumers =======================
    const int t = tid - 64;
    const int cw = warp - 2;
    bool ok = true;
    Ring rg;
    // Deferred end of a first-phase item (taken after the first stage of the
    // next item, or at the end of the phase): partial Gram (both stacked
    // blocks) to the workspace, arrival, and the Gram-space step if it
    // completed its matrix.
    auto finish = [&](int item, int k) {
      const int g = k & 1;
      const int mat = item / p.nb;
      const bool gok = mwait_warp(&B->gram_full[g], (k >> 1) & 1, ctx);
      ptx::tc_fence_after();
      const int nblk = stack ? 2 : 1;
      if (gok && ok && warp >= 4 && warp <= 7 && (warp - 4) * 32 < nblk * p.mr) {
        // stacked chunks: block bb is row block bb's diagonal block; precise:
        // row L's partial is D[L][j] + D[L][mr + j] (hi and lo columns), and
        // the two row blocks are summed with the other partials
        // lane L holds row L of D: block b = L / mr, row i = L - b mr, whose
        // diagonal block starts at column b mr
        const int L = (warp - 4) * 32 + lane;
        const int bb = L >= p.mr ? 1 : 0, i = L - bb * p.mr;
        float* dstp = p.part + static_cast<size_t>(item) * p.pstride + bb * m * m;
        const uint32_t lbase = tmem + p.gcols * g + (static_cast<uint32_t>((warp - 4) * 32) << 16);
        for (int c0 = 0; c0 < m; c0 += 32) {
          uint32_t r0[32], r1[32];
          ptx::tmem_ld_32x32b_x32(lbase + c0, r0);
          if (stack) ptx::tmem_ld_32x32b_x32(lbase + p.mr + c0, r1);
          ptx::tmem_ld_wait();
          if (L < nblk * p.mr && i < m) {
#pragma unroll
            for (int j = 0; j < 32; ++j)
              if (c0 + j < m)
                __stcg(dstp + i * m + c0 + j,
                       PRECISE ? __uint_as_float(r0[j]) + __uint_as_float(r1[j])
                                 : __uint_as_float(bb ? r1[j] : r0[j]));
          }
        }
      }
      ok = ok && gok;
      // the item's image and partial must be visible before the arrival
      __threadfence();
      ptx::tc_fence_before();
      cons_sync();
      if (t == 0)
        B->last = (ok && !B->abort &&
                   atomicAdd(larr + mat, 1u) + 1u == static_cast<unsigned>(p.nb)) ? 1 : 0;
      cons_sync();
      if (B->last) {
        __threadfence();
        if (p.mp == 32) gram_space<2, 2, 32, false>(p, mat, gs, t);
        else if (p.gs_lowmem) gram_space<4, 4, 64, true>(p, mat, gs, t);
        else gram_space<4, 4, 64, false>(p, mat, gs, t);
        __threadfence();
        cons_sync();
        // publish: next free position of the ready list (the testing hook
        // withholds the launch's last matrix, so the waits for it run out)
        if (t == 0 && !(p.inject && mat == p.total_mats - 1)) {
          const unsigned pos = atomicAdd(lctr, 1u);
          if (pos < static_cast<unsigned>(p.total_mats))
            st_release_u64(p.ready_list + pos, (static_cast<unsigned long long>(p.epoch) << 32) |
                                                   static_cast<unsigned>(mat));
        }
        cons_sync();
      }
    };
    // this warp is done with the current stage; `wrote`: it wrote the stage
    // (the first phase's X0 tile), which the tensor core then reads through
    // the async proxy; the second phase only reads it
    auto release = [&](bool wrote) {
      if (wrote) ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(&B->cons_done[rg.stage]);
      rg.next(NS);
    };
    float* escr = reinterpret_cast<float*>(sm + p.off_epi) + (warp - 2) * 128;
    int prev = -1, prevk = 0, k = 0;
    // ---- first phase ----
    for (;; ++k) {
      // One thread takes the per-item decision (next item, end, abort) so
      // that every consumer warp runs the same sequence of named barriers.
      if (t == 0) {
        int it = -2;
        if (mwait(&B->ring_full[rg.stage], rg.phase, ctx))
          it = B->desc[rg.stage][0] == kStageP1End ? -1 : B->desc[rg.stage][1];
        B->cur_item = it;
      }
      cons_sync();
      const int item = B->cur_item;
      if (item == -2) {
        ok = false;
        break;
      }
      if (item < 0) {   // end of the first phase
        mwait_warp(&B->ring_full[rg.stage], rg.phase, ctx);
        release(false);
        break;
      }
      const ItemCfg ic = item_cfg(p, item);
      for (int s = 0; s < s1; ++s) {
        const bool sok = mwait_warp(&B->ring_full[rg.stage], rg.phase, ctx);
        ok = ok && sok;
        if (ok) consume_p1_dt<PRECISE>(ic, s * p.cw1, ring + rg.stage * p.stage_bytes, t);
        release(true);
        // the previous item ends one stage into this one (its last MMAs
        // have run meanwhile): its matrix must not wait for this item
        if (s == 0 && prev >= 0) {
          finish(prev, prevk);
          prev = -1;
        }
      }
      prev = item;
      prevk = k;
    }
    if (prev >= 0) finish(prev, prevk);
    // ---- second phase: every stage until the end token ----
    // The two sets of four warps take alternate stages, so each tile's fixed
    // costs (waits, fences, the stage hand-back) are paid by half of the
    // warps while the other half works on the next tile; the other set hands
    // the stage back at once.
    const int q4 = warp & 3, set = cw >> 2;
    int cur = -1;
    ItemCfg ic{};
    for (unsigned seq = 0; ok; ++seq) {
      if (!mwait_warp(&B->ring_full[rg.stage], rg.phase, ctx)) break;
      const int kind = B->desc[rg.stage][0];
      if (kind == kStageEnd) break;
      if (static_cast<int>(seq % kSets) != set) {
        release(false);
        continue;
      }
      const int item = B->desc[rg.stage][1];
      if (item != cur) {
        cur = item;
        ic = item_cfg(p, item);
      }
      const bool sok = mwait_warp(&B->mma_done[rg.stage], rg.phase, ctx);
      ok = ok && sok;
      ptx::tc_fence_after();
      if (ok) {
        epi_tile_any(ic, B->desc[rg.stage][2], ring + rg.stage * p.stage_bytes,
                     tmem + obase + oslot_cols * rg.stage, set, q4, lane, escr,
                     &B->st_w[rg.stage], ctx);
      }
      release(false);
    }
    // the set's TMA stores have written global memory before the CTA exits
    if (q4 == 0 && lane == 0) ptx::bulk_wait_all();
  }
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) ptx::tmem_dealloc(tmem, kSmallTmemCols);
}

int small_blocks_per_sm(int smem_bytes, bool precise) {
  auto kern = precise ? ns_small_kernel<true> : ns_small_kernel<false>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  int nb = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&nb, kern, kSmallThreads, smem_bytes) !=
      cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return nb;
}

cudaError_t launch_small(const SmallParams& p, int grid, cudaStream_t s) {
  if (p.items <= 0 || grid <= 0) return cudaSuccess;
  auto kern = p.precise ? ns_small_kernel<true> : ns_small_kernel<false>;
  cudaError_t e =
      cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kSmallThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = s;
  // The second phase waits on results of other CTAs' first phase: every CTA
  // must be resident.
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace muon
