// Tensor-core GEMMs of one Newton-Schulz step (HyperParallel-FSDP section 2.3,
// Eq. (1), evaluated as A = X X^T; B' = b*A + c*A^2 + alpha*I;
// X' = (a - alpha)*X + B' X):
//
//   Gram   A  = X X^T        symmetric: only tiles holding an element with
//                            col >= row are computed, each such element is
//                            written at (r, c) and mirrored to (c, r)
//                            (DMuon-2 section 5, symmetric products);
//                            split-K over the long side for few tiles.
//   Poly   B' = b*A + c*A A + alpha*I   A is symmetric, so A A = A A^T: the
//                            same K-major operands as the Gram; the rest is
//                            fused in the epilogue; symmetric output.
//   Apply  X'^T = (a - alpha)*X^T + X^T B'   (B' symmetric), i.e.
//                            X' = (a - alpha)*X + B' X; writes both layouts
//                            of X' (the next Gram reads X, the next Apply X^T).
//
// Every product is D = P Q^T with P and Q K-major bf16 in global memory, so
// one persistent kernel body serves all three.  Per CTA (one per SM):
//   warp 0      TMA producer: 128x64 (P) and 256x64 (Q) tiles, 128-byte
//               swizzle, into a 4-stage shared-memory ring;
//   warp 1      allocates TMEM and issues tcgen05.mma (M=128, N=256, K=16)
//               from one elected thread into one of two TMEM accumulators;
//   warps 2..5  epilogue: tcgen05.ld, fused arithmetic, 16-byte stores; the
//               transposed / mirrored copies go through a per-warp
//               shared-memory transpose so they are written as whole rows.
// The two accumulators let the epilogue of tile t overlap the mainloop of
// tile t+1.  Tiles of all matrices of all core-shape groups of a chunk form
// one static round-robin schedule.  Every wait is bounded; on a timeout a
// status bit is set, in-flight copies are drained, TMEM is freed and the CTA
// returns.
#include "muon_internal.h"
#include "sm100_ptx.cuh"

namespace muon {

namespace {

constexpr int BM = 128;          // MMA M = TMEM lanes
constexpr int BN = 256;          // MMA N = TMEM columns per accumulator
constexpr int BK = 64;           // one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;       // K per tcgen05.mma (kind::f16)
constexpr int kStages = 4;
constexpr int kABytes = BM * BK * 2;
constexpr int kBBytes = BN * BK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kThreads = 192;
constexpr int kEpiWarp0 = 2;
constexpr int kTpitch = 40;      // bf16 pitch of a 32x32 transpose block (80 B rows)
constexpr int kTBytes = 32 * kTpitch * 2;
constexpr int kBarOff = kStages * kStageBytes + 4 * kTBytes;
constexpr int kSmemBytes = kBarOff + 256 + 1024;
constexpr uint32_t kTmemCols = 2 * BN;

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

__device__ __forceinline__ void epi_bar() {   // the four epilogue warps only
  asm volatile("bar.sync 1, 128;" ::: "memory");
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

template <int EPI>
__device__ __forceinline__ TileInfo decode(const GemmParams& p, int tile) {
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
    t.row_tile = r / G.nt;
    t.col_tile = r - t.row_tile * G.nt;
  } else {
    int idx = r / G.ksplit;
    t.ksp = r - idx * G.ksplit;
    t.sym_idx = idx;
    int j = 0;
    for (;;) {
      const int c = sym_rows(j, G.mt);
      if (idx < c) break;
      idx -= c;
      ++j;
    }
    t.row_tile = idx;
    t.col_tile = j;
  }
  t.kb0 = t.ksp * G.kb_per_split;
  const int e = t.kb0 + G.kb_per_split < G.num_kb ? t.kb0 + G.kb_per_split : G.num_kb;
  t.nkb = e - t.kb0;
  return t;
}

__device__ __forceinline__ void ld_bf16x32(const __nv_bfloat16* p, float* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const uint4 u = *reinterpret_cast<const uint4*>(p + 8 * q);
    const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float2 f = __bfloat1622float2(h[k]);
      v[8 * q + 2 * k] = f.x;
      v[8 * q + 2 * k + 1] = f.y;
    }
  }
}

__device__ __forceinline__ void st_bf16x32(__nv_bfloat16* p, const __nv_bfloat16* v) {
#pragma unroll
  for (int q = 0; q < 4; ++q)
    *reinterpret_cast<uint4*>(p + 8 * q) = *reinterpret_cast<const uint4*>(v + 8 * q);
}

// Write the warp's 32x32 block transposed: lane l owns row (r0 + l) of the
// block and the 32 values h[0..31] at columns c0..c0+31; afterwards lane l
// writes column (c0 + l) as a row of 32 values at dst + (c0 + l)*pitch + r0.
// Elements outside [0, rows_lim) x [0, cols_lim) are skipped, and when
// `upper_only` is set only elements with column > row are written.
__device__ __forceinline__ void store_transposed(__nv_bfloat16* tb, const __nv_bfloat16* h,
                                                 __nv_bfloat16* dst, int64_t pitch, int64_t r0,
                                                 int64_t c0, int64_t rows_lim, int64_t cols_lim,
                                                 bool upper_only) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int j = 0; j < 32; ++j) tb[j * kTpitch + lane] = h[j];
  __syncwarp();
  const int64_t c = c0 + lane;                 // row of dst
  const __nv_bfloat16* src = tb + lane * kTpitch;
  const bool full = (r0 + 32 <= rows_lim) && (!upper_only || c0 > r0 + 31);
  if (c < cols_lim) {
    __nv_bfloat16* d = dst + c * pitch + r0;
    if (full) {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        *reinterpret_cast<uint4*>(d + 8 * q) = *reinterpret_cast<const uint4*>(src + 8 * q);
    } else {
      for (int k = 0; k < 32; ++k) {
        const int64_t r = r0 + k;
        if (r < rows_lim && (!upper_only || c > r)) d[k] = src[k];
      }
    }
  }
  __syncwarp();
}

}  // namespace

template <int EPI>
__global__ void __launch_bounds__(kThreads, 1) ns_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  __nv_bfloat16* sT = reinterpret_cast<__nv_bfloat16*>(smem + kStages * kStageBytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kBarOff);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;      // [2] accumulator ready
  uint64_t* tempty = tfull + 2;           // [2] accumulator drained
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(tempty + 2);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_last = reinterpret_cast<int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      ptx::mbar_init(&tfull[b], 1);
      ptx::mbar_init(&tempty[b], 128);
    }
    *abort_flag = 0;
    ptx::fence_mbar_init();
    for (int g = 0; g < p.n_groups; ++g) {
      ptx::prefetch_tmap(&p.g[g].mapA);
      ptx::prefetch_tmap(&p.g[g].mapB);
    }
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- TMA producer ------------------------------------------------------------------
    if (lane == 0) {
      int stage = 0, issued = 0;
      uint32_t phase = 0;
      bool stop = false;
      for (int tile = blockIdx.x; tile < p.total_tiles && !stop; tile += gridDim.x) {
        const TileInfo t = decode<EPI>(p, tile);
        const GemmGroup& G = p.g[t.gi];
        for (int i = 0; i < t.nkb; ++i) {
          if (!wait_bounded(&empty[stage], phase ^ 1, abort_flag, p.status, p.timeout_ns, true)) {
            stop = true;
            break;
          }
          ptx::mbar_arrive_expect_tx(&full[stage], kStageBytes);
          const int kx = (t.kb0 + i) * BK;
          ptx::tma_load_3d(sA + stage * kABytes, &G.mapA, &full[stage], kx, t.row_tile * BM, t.mat);
          ptx::tma_load_3d(sB + stage * kBBytes, &G.mapB, &full[stage], kx, t.col_tile * BN, t.mat);
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
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN);
      int stage = 0, acc = 0;
      uint32_t phase = 0;
      bool stop = false;
      for (int tile = blockIdx.x; tile < p.total_tiles && !stop; tile += gridDim.x, ++acc) {
        const TileInfo t = decode<EPI>(p, tile);
        const int buf = acc & 1;
        if (!wait_bounded(&tempty[buf], ((acc >> 1) & 1) ^ 1, abort_flag, p.status, p.timeout_ns,
                          true)) {
          stop = true;
          break;
        }
        ptx::tc_fence_after();
        const uint32_t d = tmem + buf * BN;
        for (int i = 0; i < t.nkb; ++i) {
          if (!wait_bounded(&full[stage], phase, abort_flag, p.status, p.timeout_ns, true)) {
            stop = true;
            break;
          }
          ptx::tc_fence_after();
          const uint32_t a0 = ptx::smem_u32(sA + stage * kABytes);
          const uint32_t b0 = ptx::smem_u32(sB + stage * kBBytes);
#pragma unroll
          for (int k = 0; k < BK / UMMA_K; ++k)
            ptx::umma_bf16(d, ptx::sdesc_kmajor_sw128(a0 + k * UMMA_K * 2),
                           ptx::sdesc_kmajor_sw128(b0 + k * UMMA_K * 2), idesc,
                           (i > 0 || k > 0) ? 1u : 0u);
          ptx::umma_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1;
          }
        }
        ptx::umma_commit(&tfull[buf]);   // accumulator complete (or abandoned)
      }
    }
    __syncwarp();
  } else {
    // ---- epilogue (warps 2..5; TMEM lane quadrant = warp % 4) ---------------------------------
    const int q4 = warp & 3;
    const int row = q4 * 32 + lane;
    __nv_bfloat16* tb = sT + (warp - kEpiWarp0) * (32 * kTpitch);
    int acc = 0;
    for (int tile = blockIdx.x; tile < p.total_tiles; tile += gridDim.x, ++acc) {
      const TileInfo t = decode<EPI>(p, tile);
      const GemmGroup& G = p.g[t.gi];
      const int buf = acc & 1;
      wait_bounded(&tfull[buf], (acc >> 1) & 1, abort_flag, p.status, p.timeout_ns, false);
      // one decision for all four epilogue warps (they share named barriers)
      epi_bar();
      const bool ok = !*abort_flag;
      ptx::tc_fence_after();
      const uint32_t taddr = tmem + buf * BN + (static_cast<uint32_t>(q4 * 32) << 16);
      if (!ok) {
        ptx::tc_fence_before();
        ptx::mbar_arrive(&tempty[buf]);
        break;
      }
      if (EPI == kEpiApply) {
        const int64_t gp = (int64_t)t.row_tile * BM + row;      // index along n
        const int64_t gp0 = (int64_t)t.row_tile * BM + q4 * 32; // first row of this warp
        const float s = p.first ? G.inv[t.mat] : 1.f;
        const __nv_bfloat16* xin = G.epi_in + (int64_t)t.mat * G.mstride_in + gp * G.pitch_in;
        __nv_bfloat16* xt_out = G.out0 + (int64_t)t.mat * G.mstride0 + gp * G.pitch0;
        __nv_bfloat16* x_out = G.out1 + (int64_t)t.mat * G.mstride1;
        for (int c0 = 0; c0 < BN; c0 += 32) {
          const int64_t gq0 = (int64_t)t.col_tile * BN + c0;   // index along m
          if (gq0 >= G.m) break;                                // warp-uniform
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(taddr + c0, r);
          ptx::tmem_ld_wait();
          const bool fullc = gq0 + 32 <= G.m;
          float x[32];
          if (gp < G.n) {
            if (fullc) {
              ld_bf16x32(xin + gq0, x);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j) x[j] = gq0 + j < G.m ? __bfloat162float(xin[gq0 + j]) : 0.f;
            }
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) x[j] = 0.f;
          }
          __align__(16) __nv_bfloat16 h[32];
#pragma unroll
          for (int j = 0; j < 32; ++j)
            h[j] = __float2bfloat16_rn(s * fmaf(p.a, x[j], __uint_as_float(r[j])));
          if (gp < G.n) {
            if (fullc) {
              st_bf16x32(xt_out + gq0, h);
            } else {
              for (int j = 0; j < 32; ++j)
                if (gq0 + j < G.m) xt_out[gq0 + j] = h[j];
            }
          }
          // X'[q][p]: rows gq0.., columns gp0..gp0+31
          store_transposed(tb, h, x_out, G.pitch1, gp0, gq0, G.n, G.m, false);
        }
        ptx::tc_fence_before();
        ptx::mbar_arrive(&tempty[buf]);
      } else {
        const int64_t gr = (int64_t)t.row_tile * BM + row;
        const int64_t gr0 = (int64_t)t.row_tile * BM + q4 * 32;
        const bool split = G.ksplit > 1;
        const int64_t slot = (int64_t)t.mat * G.tiles_per_mat / G.ksplit + t.sym_idx;
        float* part = split ? G.partial + slot * G.ksplit * (int64_t)(BM * BN) : nullptr;
        if (split) {
          // partial tile -> global (valid entries only), then the last split reduces
          for (int c0 = 0; c0 < BN; c0 += 32) {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(taddr + c0, r);
            ptx::tmem_ld_wait();
            if (gr < G.m) {
#pragma unroll
              for (int j = 0; j < 32; ++j) {
                const int64_t gc = (int64_t)t.col_tile * BN + c0 + j;
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
        const float scale = (EPI == kEpiGram && p.first) ? G.inv[t.mat] * G.inv[t.mat] : 1.f;
        __nv_bfloat16* out = G.out0 + (int64_t)t.mat * G.mstride0;
        const __nv_bfloat16* ain =
            (EPI == kEpiPoly) ? G.epi_in + (int64_t)t.mat * G.mstride_in : nullptr;
        for (int c0 = 0; c0 < BN; c0 += 32) {
          const int64_t gc0 = (int64_t)t.col_tile * BN + c0;
          if (gc0 >= G.m) break;                               // warp-uniform
          if (gc0 + 31 < gr0) continue;                        // block entirely below the diagonal
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
          const bool fullc = gc0 + 32 <= G.m;
          float av[32];
          if (EPI == kEpiPoly) {
            if (gr < G.m && fullc) {
              ld_bf16x32(ain + gr * G.pitch_in + gc0, av);
            } else {
#pragma unroll
              for (int j = 0; j < 32; ++j)
                av[j] = (gr < G.m && gc0 + j < G.m) ? __bfloat162float(ain[gr * G.pitch_in + gc0 + j])
                                                    : 0.f;
            }
          }
          __align__(16) __nv_bfloat16 h[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            float val = v[j] * scale;
            if (EPI == kEpiPoly)
              val = fmaf(p.b, av[j], p.c * val) + (gr == gc0 + j ? p.alpha : 0.f);
            h[j] = __float2bfloat16_rn(val);
          }
          // direct (r, c) for c >= r
          if (gr < G.m) {
            __nv_bfloat16* o = out + gr * G.pitch0 + gc0;
            if (fullc && gc0 >= gr) {
              st_bf16x32(o, h);
            } else {
              for (int j = 0; j < 32; ++j)
                if (gc0 + j < G.m && gc0 + j >= gr) o[j] = h[j];
            }
          }
          // mirror (c, r) for c > r
          store_transposed(tb, h, out, G.pitch0, gr0, gc0, G.m, G.m, true);
        }
        if (!split) {
          ptx::tc_fence_before();
          ptx::mbar_arrive(&tempty[buf]);
        } else if (threadIdx.x == kEpiWarp0 * 32) {
          G.tile_cnt[slot] = 0u;
        }
      }
    }
  }

  ptx::tc_fence_before();
  __syncthreads();
  if (warp == 1) ptx::tmem_dealloc(tmem, kTmemCols);
}

int gemm_block_n() { return BN; }
int gemm_block_m() { return BM; }
int gemm_block_k() { return BK; }

int gemm_sym_tiles(int m) {
  const int ntr = (m + BM - 1) / BM, ntc = (m + BN - 1) / BN;
  int t = 0;
  for (int j = 0; j < ntc; ++j) {
    const int r = (BN * j + BN - 1) / BM + 1;
    t += r < ntr ? r : ntr;
  }
  return t;
}

template <int EPI>
static cudaError_t launch_one(const GemmParams& p, int grid, cudaStream_t s) {
  cudaError_t e = cudaFuncSetAttribute(ns_gemm_kernel<EPI>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
  if (e != cudaSuccess) return e;
  ns_gemm_kernel<EPI><<<grid, kThreads, kSmemBytes, s>>>(p);
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
  switch (epi) {
    case kEpiGram: return launch_one<kEpiGram>(p, grid, s);
    case kEpiPoly: return launch_one<kEpiPoly>(p, grid, s);
    case kEpiApply: return launch_one<kEpiApply>(p, grid, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace muon
