// Tensor-core GEMMs of one Newton-Schulz step (HyperParallel-FSDP section 2.3,
// Eq. (1), evaluated as A = X X^T; B = b*A + c*A^2; X' = a*X + B X):
//
//   Gram   A  = X X^T        symmetric: only tiles (i <= j) are computed and
//                            mirrored (DMuon-2 section 5, symmetric products);
//                            split-K over the long side for tall-skinny X.
//   Poly   B  = b*A + c*A A  A is symmetric, so A A = A A^T: same K-major
//                            operands as the Gram; b*A + c*(.) fused in the
//                            epilogue; symmetric output.
//   Apply  X'^T = a*X^T + X^T B   (B symmetric), i.e. X' = a*X + B X,
//                            with a*X fused in the epilogue; writes both
//                            layouts of X' (the next Gram reads X, the next
//                            Apply reads X^T).
//
// Every product is D = P Q^T with P and Q K-major bf16 in global memory, so a
// single kernel body serves all three: TMA (128-byte swizzle) stages P and Q
// tiles into a shared-memory ring, one elected thread issues tcgen05.mma into
// a TMEM accumulator, and four warps drain TMEM with tcgen05.ld for the fused
// epilogue.  A launch covers all matrices of all core-shape groups of a chunk
// (a grouped tile table), so a step issues a fixed number of launches however
// many matrices it has.  Every wait is bounded; a timeout sets a status bit
// and the CTA drains its in-flight copies, frees TMEM and returns.
#include "muon_internal.h"
#include "sm100_ptx.cuh"

namespace muon {

namespace {

constexpr int BM = 128;          // MMA M = TMEM lanes
constexpr int BN = 128;          // MMA N = TMEM columns
constexpr int BK = 64;           // one 128-byte swizzle row of bf16
constexpr int UMMA_K = 16;       // K per tcgen05.mma (kind::f16)
constexpr int kStages = 3;
constexpr int kABytes = BM * BK * 2;
constexpr int kBBytes = BN * BK * 2;
constexpr int kStageBytes = kABytes + kBBytes;
constexpr int kSmemBytes = kStages * kStageBytes + 1024 /*align*/ + 256 /*barriers*/;
constexpr uint32_t kTmemCols = BN;

__device__ __forceinline__ bool wait_bounded(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, unsigned* status,
                                             unsigned long long timeout_ns,
                                             bool honour_abort) {
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

__device__ __forceinline__ void tri_decode(int idx, int nt, int& i, int& j) {
  i = 0;
  while (idx >= nt - i) {
    idx -= nt - i;
    ++i;
  }
  j = i + idx;
}

}  // namespace

template <int EPI>
__global__ void __launch_bounds__(128, 1) ns_gemm_kernel(const __grid_constant__ GemmParams p) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t base_u32 = ptx::smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (base_u32 & 1023u)) & 1023u);
  uint8_t* sA = smem;
  uint8_t* sB = smem + kStages * kABytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * kStageBytes);
  uint64_t* empty = full + kStages;
  uint64_t* done = empty + kStages;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(done + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  int* s_last = reinterpret_cast<int*>(tmem_slot + 2);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // ---- decode the tile ---------------------------------------------------------
  const int tile = blockIdx.x;
  int gi = 0;
  while (gi + 1 < p.n_groups && tile >= p.g[gi + 1].tile_base) ++gi;
  const GemmGroup& G = p.g[gi];
  const int local = tile - G.tile_base;
  const int mat = local / G.tiles_per_mat;
  const int t = local - mat * G.tiles_per_mat;
  int row_tile, col_tile, ksp = 0, tri = 0;
  if (EPI == kEpiApply) {
    row_tile = t / G.nt;
    col_tile = t - row_tile * G.nt;
  } else {
    tri = t / G.ksplit;
    ksp = t - tri * G.ksplit;
    tri_decode(tri, G.nt, row_tile, col_tile);
  }
  const int kb0 = ksp * G.kb_per_split;
  const int nkb = min(G.num_kb, kb0 + G.kb_per_split) - kb0;
  const bool diag = (EPI != kEpiApply) && (row_tile == col_tile);

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      ptx::mbar_init(&full[s], 1);
      ptx::mbar_init(&empty[s], 1);
    }
    ptx::mbar_init(done, 1);
    *abort_flag = 0;
    ptx::fence_mbar_init();
    ptx::prefetch_tmap(&G.mapA);
    ptx::prefetch_tmap(&G.mapB);
  }
  if (warp == 1) ptx::tmem_alloc(tmem_slot, kTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ---- TMA producer ----------------------------------------------------------
    if (lane == 0) {
      const uint32_t tx = diag ? kABytes : kABytes + kBBytes;
      int issued = 0;
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!wait_bounded(&empty[s], ph ^ 1, abort_flag, p.status, p.timeout_ns, true)) break;
        ptx::mbar_arrive_expect_tx(&full[s], tx);
        const int kx = (kb0 + i) * BK;
        ptx::tma_load_3d(sA + s * kABytes, &G.mapA, &full[s], kx, row_tile * BM, mat);
        if (!diag) ptx::tma_load_3d(sB + s * kBBytes, &G.mapB, &full[s], kx, col_tile * BN, mat);
        ++issued;
      }
      // drain: every issued copy has landed before this CTA may exit
      for (int j = max(0, issued - kStages); j < issued; ++j)
        wait_bounded(&full[j % kStages], (j / kStages) & 1, abort_flag, p.status, p.timeout_ns,
                     false);
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---- MMA issuer ------------------------------------------------------------
    if (lane == 0) {
      constexpr uint32_t idesc = ptx::idesc_bf16_f32(BM, BN);
      for (int i = 0; i < nkb; ++i) {
        const int s = i % kStages;
        const uint32_t ph = (i / kStages) & 1;
        if (!wait_bounded(&full[s], ph, abort_flag, p.status, p.timeout_ns, true)) break;
        ptx::tc_fence_after();
        const uint32_t a0 = ptx::smem_u32(sA + s * kABytes);
        const uint32_t b0 = diag ? a0 : ptx::smem_u32(sB + s * kBBytes);
#pragma unroll
        for (int k = 0; k < BK / UMMA_K; ++k) {
          ptx::umma_bf16(tmem, ptx::sdesc_kmajor_sw128(a0 + k * UMMA_K * 2),
                         ptx::sdesc_kmajor_sw128(b0 + k * UMMA_K * 2), idesc,
                         (i > 0 || k > 0) ? 1u : 0u);
        }
        ptx::umma_commit(&empty[s]);   // frees the stage once these MMAs are done
      }
      ptx::umma_commit(done);          // accumulator complete (or abandoned)
    }
    __syncwarp();
  }

  // ---- epilogue: all four warps, TMEM lane = tile row ----------------------------
  const bool ok = wait_bounded(done, 0, abort_flag, p.status, p.timeout_ns, false) && !*abort_flag;
  ptx::tc_fence_after();
  const int row = warp * 32 + lane;
  const uint32_t taddr = tmem + (static_cast<uint32_t>(warp * 32) << 16);

  if (ok) {
    if (EPI == kEpiApply) {
      const int64_t gp = (int64_t)row_tile * BM + row;     // index along n
      const float s = p.first ? G.inv[mat] : 1.f;
      const __nv_bfloat16* xin = G.epi_in + (int64_t)mat * G.mstride_in + gp * G.pitch_in;
      __nv_bfloat16* xt_out = G.out0 + (int64_t)mat * G.mstride0 + gp * G.pitch0;
      __nv_bfloat16* x_out = G.out1 + (int64_t)mat * G.mstride1 + gp;
      for (int c0 = 0; c0 < BN; c0 += 32) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(taddr + c0, r);
        ptx::tmem_ld_wait();
        if (gp < G.n) {
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int64_t gq = (int64_t)col_tile * BN + c0 + j;   // index along m
            if (gq < G.m) {
              const float x = __bfloat162float(xin[gq]);
              const __nv_bfloat16 v = __float2bfloat16_rn(s * fmaf(p.a, x, __uint_as_float(r[j])));
              xt_out[gq] = v;
              x_out[gq * G.pitch1] = v;
            }
          }
        }
      }
    } else {
      const int64_t gr = (int64_t)row_tile * BM + row;
      const bool split = G.ksplit > 1;
      const int tri_tiles = G.nt * (G.nt + 1) / 2;
      const int64_t slot = (int64_t)mat * tri_tiles + tri;
      float* part = split ? G.partial + (slot * G.ksplit) * (int64_t)(BM * BN) : nullptr;
      if (split) {
        for (int c0 = 0; c0 < BN; c0 += 32) {
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(taddr + c0, r);
          ptx::tmem_ld_wait();
          if (gr < G.m) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int64_t gc = (int64_t)col_tile * BN + c0 + j;
              if (gc < G.m)
                __stcg(part + (int64_t)ksp * (BM * BN) + (c0 + j) * BM + row,
                       __uint_as_float(r[j]));
            }
          }
        }
        __threadfence();
        __syncthreads();
        if (threadIdx.x == 0) {
          const unsigned prev = atomicAdd(&G.tile_cnt[slot], 1u);
          *s_last = (prev == (unsigned)(G.ksplit - 1));
        }
        __syncthreads();
        __threadfence();
      }
      if (!split || *s_last) {
        const float scale = (EPI == kEpiGram && p.first) ? G.inv[mat] * G.inv[mat] : 1.f;
        __nv_bfloat16* out = G.out0 + (int64_t)mat * G.mstride0;
        const __nv_bfloat16* ain = (EPI == kEpiPoly) ? G.epi_in + (int64_t)mat * G.mstride_in
                                                     : nullptr;
        for (int c0 = 0; c0 < BN; c0 += 32) {
          float v[32];
          if (split) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              float acc = 0.f;
              const int64_t gc = (int64_t)col_tile * BN + c0 + j;
              if (gr < G.m && gc < G.m)
                for (int q = 0; q < G.ksplit; ++q)
                  acc += __ldcg(part + (int64_t)q * (BM * BN) + (c0 + j) * BM + row);
              v[j] = acc;
            }
          } else {
            uint32_t r[32];
            ptx::tmem_ld_32x32b_x32(taddr + c0, r);
            ptx::tmem_ld_wait();
#pragma unroll
            for (int j = 0; j < 32; ++j) v[j] = __uint_as_float(r[j]);
          }
          if (gr < G.m) {
#pragma unroll
            for (int j = 0; j < 32; ++j) {
              const int64_t gc = (int64_t)col_tile * BN + c0 + j;
              if (gc < G.m && (row_tile < col_tile || gc >= gr)) {
                float val = v[j] * scale;
                if (EPI == kEpiPoly)
                  val = fmaf(p.b, __bfloat162float(ain[gr * G.pitch_in + gc]), p.c * val) +
                        (gr == gc ? p.alpha : 0.f);
                const __nv_bfloat16 h = __float2bfloat16_rn(val);
                out[gr * G.pitch0 + gc] = h;
                out[gc * G.pitch0 + gr] = h;
              }
            }
          }
        }
        if (split && threadIdx.x == 0) G.tile_cnt[slot] = 0u;
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

template <int EPI>
static cudaError_t launch_one(const GemmParams& p, cudaStream_t s) {
  static bool attr_set = false;
  if (!attr_set) {
    cudaError_t e = cudaFuncSetAttribute(ns_gemm_kernel<EPI>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemBytes);
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  ns_gemm_kernel<EPI><<<p.total_tiles, 128, kSmemBytes, s>>>(p);
  return cudaGetLastError();
}

cudaError_t launch_gemm(int epi, const GemmParams& p, cudaStream_t s) {
  if (p.total_tiles <= 0) return cudaSuccess;
  switch (epi) {
    case kEpiGram: return launch_one<kEpiGram>(p, s);
    case kEpiPoly: return launch_one<kEpiPoly>(p, s);
    case kEpiApply: return launch_one<kEpiApply>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace muon
