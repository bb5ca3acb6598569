// Fused Muon step for matrices with a small side (m <= 64 after the
// transpose-first rule), one thread-block cluster per matrix.
//
// HyperParallel-FSDP section 6.6 and RFC issue 204 item 3 fuse many small
// matrices of one core shape into one batched launch because per-matrix
// launches starve the device; this kernel goes one step further and runs the
// whole step of a matrix -- momentum, norm, every Newton-Schulz iteration and
// the update -- in one launch, with X resident in the distributed shared
// memory of a cluster of `cs` CTAs (CTA r holds columns [r*w, (r+1)*w) of X).
//
// Shared-memory layout of X (one layout serves both products): chunks of 64
// columns, each chunk mr rows x 128 bytes with the 128-byte swizzle.
//   Gram   A = X X^T: K-major view (rows = m, K = columns); M = 128 rows are
//          issued, rows >= m read neighbouring memory and are ignored.  Each
//          CTA forms its partial over its columns; the partials are summed in
//          rank order over DSMEM after a cluster barrier, identically in every
//          CTA.
//   Poly   P = a*I + b*A + c*A^2 on CUDA cores (m^3 <= 262144 MACs), in fp32
//          from the fp32 A, stored as two bf16 K-major MMA operands P = hi + lo
//          (the apply issues both), so neither A nor P is rounded to bf16 as
//          a whole; X' = a*X + (b*A + c*A^2)*X = P*X.
//   Apply  X'^T = X^T P: the A operand is the MN-major view of the same X
//          chunks (M = 128 columns of X, K = m), P the K-major B operand;
//          the epilogue only converts and writes X' back in place.
// Rows >= m of P and its columns >= m are zero, so the K padding of the
// apply contributes nothing.  The two P tiles (hi at +0, lo at +8 KB) also
// serve as the landing zone of the Gram's ignored rows past the last chunk.
#include "muon_internal.h"
#include "sm100_ptx.cuh"

namespace muon {

namespace {

__device__ __forceinline__ bool wait_mma(uint64_t* bar, uint32_t parity, unsigned* status,
                                         unsigned long long timeout_ns) {
  const uint32_t addr = ptx::smem_u32(bar);
  if (ptx::mbar_try_wait(addr, parity)) return true;
  const uint64_t t0 = ptx::globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (ptx::mbar_try_wait(addr, parity)) return true;
    if ((it & 255u) == 0 && ptx::globaltimer() - t0 > timeout_ns) {
      atomicOr(status, kDevTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ void load8(const void* base, int dtype, int64_t e, int nvalid, bool vec,
                                      float* d) {
  if (vec && nvalid == 8) {
    if (dtype == 0) {
      const float4 a = __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(base) + e));
      const float4 b =
          __ldcs(reinterpret_cast<const float4*>(static_cast<const float*>(base) + e + 4));
      d[0] = a.x; d[1] = a.y; d[2] = a.z; d[3] = a.w;
      d[4] = b.x; d[5] = b.y; d[6] = b.z; d[7] = b.w;
    } else {
      const uint4 u = __ldcs(
          reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(base) + e));
      const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&u);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(h[j]);
        d[2 * j] = f.x;
        d[2 * j + 1] = f.y;
      }
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    float v = 0.f;
    if (j < nvalid)
      v = dtype == 0 ? static_cast<const float*>(base)[e + j]
                     : __bfloat162float(static_cast<const __nv_bfloat16*>(base)[e + j]);
    d[j] = v;
  }
}

__device__ __forceinline__ void store8(void* base, int dtype, int64_t e, int nvalid, bool vec,
                                       const float* d) {
  if (vec && nvalid == 8) {
    if (dtype == 0) {
      float* f = static_cast<float*>(base) + e;
      *reinterpret_cast<float4*>(f) = make_float4(d[0], d[1], d[2], d[3]);
      *reinterpret_cast<float4*>(f + 4) = make_float4(d[4], d[5], d[6], d[7]);
    } else {
      uint4 u;
      __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&u);
#pragma unroll
      for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(d[2 * j], d[2 * j + 1]);
      *reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(base) + e) = u;
    }
    return;
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    if (j < nvalid) {
      if (dtype == 0) static_cast<float*>(base)[e + j] = d[j];
      else static_cast<__nv_bfloat16*>(base)[e + j] = __float2bfloat16_rn(d[j]);
    }
  }
}

}  // namespace

__global__ void __launch_bounds__(kSmallThreads, 2)
    ns_small_kernel(const __grid_constant__ SmallParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* sm = smem_raw + ((1024u - (ptx::smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sX = sm;
  uint8_t* sBt = sm + p.off_bt;
  float* sP = reinterpret_cast<float*>(sm + p.off_part);   // [2][m*m]
  float* sA = reinterpret_cast<float*>(sm + p.off_a);      // [m][m+1]
  uint64_t* bar = reinterpret_cast<uint64_t*>(sm + p.off_misc);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(bar + 1);
  float* red = reinterpret_cast<float*>(tslot + 4);          // [8]
  float* s_ssq = red + 8;
  float* s_inv = red + 9;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const uint32_t rank = ptx::cluster_ctarank();
  const int mat = blockIdx.x / p.cs;
  int si = 0;
  while (si + 1 < p.n_slices && mat >= p.s[si + 1].mat_base) ++si;
  const SmallSlice& S = p.s[si];
  const int local = mat - S.mat_base;
  const int m = p.m, n = p.n, w = p.w;
  const int64_t col0 = static_cast<int64_t>(rank) * w;
  const int chunk_bytes = p.mr * 128;
  const int nchunks = w / 64;
  const int64_t mn = static_cast<int64_t>(m) * n;

  // X (with its padding) and the B' tile start at zero.
  for (int i = tid; i < p.off_part / 16; i += kSmallThreads)
    reinterpret_cast<uint4*>(sm)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
  }
  if (warp == 0) ptx::tmem_alloc(tslot, kSmallTmemCols);
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = *tslot;

  // ---- momentum + Nesterov + cast into the cluster-resident X -------------------
  // X[i][j] = D[i][j] (stored [m][n]) or D[j][i] (stored [n][m], transposed).
  float ssq = 0.f;
  const int64_t moff = static_cast<int64_t>(local) * mn;
  // Items are 8 consecutive stored elements; each thread keeps kSmallUnroll
  // items' loads in flight before using them.
  const int ig = (m + 7) / 8;
  const int items = S.trans ? w * ig : m * (w / 8);
  for (int base = tid; base < items; base += kSmallUnroll * kSmallThreads) {
    float g[kSmallUnroll][8], mo[kSmallUnroll][8];
    int64_t e[kSmallUnroll];
    int nv[kSmallUnroll], row[kSmallUnroll], jl[kSmallUnroll];
#pragma unroll
    for (int u = 0; u < kSmallUnroll; ++u) {
      const int item = base + u * kSmallThreads;
      nv[u] = 0;
      if (item < items) {
        if (!S.trans) {
          const int gpr = w / 8;
          row[u] = item / gpr;
          jl[u] = (item - row[u] * gpr) * 8;
          const int64_t gj = col0 + jl[u];
          if (gj < n) {
            nv[u] = (n - gj) < 8 ? static_cast<int>(n - gj) : 8;
            e[u] = moff + static_cast<int64_t>(row[u]) * n + gj;
          }
        } else {
          jl[u] = item / ig;
          row[u] = (item - jl[u] * ig) * 8;
          const int64_t gj = col0 + jl[u];
          if (gj < n) {
            nv[u] = min(8, m - row[u]);
            e[u] = moff + gj * m + row[u];
          }
        }
      }
      if (nv[u] > 0) {
        load8(S.G, S.g_dtype, e[u], nv[u], S.gvec, g[u]);
        if (p.step_mode) load8(S.Mom, 0, e[u], nv[u], S.gvec, mo[u]);
      }
    }
#pragma unroll
    for (int u = 0; u < kSmallUnroll; ++u) {
      if (nv[u] <= 0) continue;
      float d[8];
      if (p.step_mode) {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          mo[u][j] = fmaf(p.mu, mo[u][j], g[u][j]);             // M_t = mu*M_{t-1} + G
          d[j] = p.nesterov ? fmaf(p.mu, mo[u][j], g[u][j]) : mo[u][j];
        }
        store8(S.Mom, 0, e[u], nv[u], S.gvec, mo[u]);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) d[j] = g[u][j];
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        if (j >= nv[u]) d[j] = 0.f;
        ssq = fmaf(d[j], d[j], ssq);
      }
      uint8_t* col = sX + (jl[u] >> 6) * chunk_bytes;
      if (!S.trans) {
        uint4 q;
        __nv_bfloat162* h = reinterpret_cast<__nv_bfloat162*>(&q);
#pragma unroll
        for (int j = 0; j < 4; ++j) h[j] = __floats2bfloat162_rn(d[2 * j], d[2 * j + 1]);
        *reinterpret_cast<uint4*>(col + ptx::sw128_offset(row[u], (jl[u] & 63) * 2)) = q;
      } else {
        const uint32_t byte = (jl[u] & 63) * 2;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < nv[u])
            *reinterpret_cast<__nv_bfloat16*>(col + ptx::sw128_offset(row[u] + j, byte)) =
                __float2bfloat16_rn(d[j]);
      }
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) ssq += __shfl_xor_sync(0xffffffffu, ssq, o);
  if (lane == 0) red[warp] = ssq;
  __syncthreads();
  if (tid == 0) {
    float b = 0.f;
    for (int i = 0; i < kSmallThreads / 32; ++i) b += red[i];
    *s_ssq = b;
  }
  ptx::fence_proxy_async_smem();
  ptx::cluster_sync();
  if (tid == 0) {
    double tot = 0.0;
    const uint32_t a = ptx::smem_u32(s_ssq);
    for (int r = 0; r < p.cs; ++r) tot += (double)ptx::ld_shared_cluster_f32(ptx::mapa_shared(a, r));
    if (!isfinite(tot) && rank == 0) atomicOr(p.status, kDevNonfinite);
    *s_inv = static_cast<float>(1.0 / (sqrt(tot) + (double)p.eps));
  }
  __syncthreads();
  const float inv = *s_inv;

  // ---- Newton-Schulz iterations -----------------------------------------------------
  const uint32_t sX_u = ptx::smem_u32(sX), sBt_u = ptx::smem_u32(sBt);
  const int nmm = p.nmm;
  const int tcol = (nmm + 31) & ~31;                 // TMEM columns per product tile
  const uint32_t idesc_gram = ptx::idesc_bf16_f32(128, nmm);
  const uint32_t idesc_app = ptx::idesc_bf16_f32(128, nmm) | (1u << 15);   // A MN-major
  const int tiles = w / 128;
  const int per_batch = (kSmallTmemCols - tcol) / tcol;
  uint32_t phase = 0;
  bool ok = true;
  for (int it = 0; it < p.steps; ++it) {
    const float ca = p.coef[it][0], cb = p.coef[it][1], cc = p.coef[it][2], al = p.coef[it][3];
    const bool first = it == 0;
    const int par = it & 1;
    // Gram partial over this CTA's columns
    if (tid == 0) {
      ptx::tc_fence_after();
      for (int kc = 0; kc < nchunks; ++kc) {
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          const uint64_t d = ptx::sdesc_kmajor_sw128(sX_u + kc * chunk_bytes + k * 32);
          ptx::umma_bf16(tmem, d, d, idesc_gram, (kc | k) != 0 ? 1u : 0u);
        }
      }
      ptx::umma_commit(bar);
    }
    __syncwarp();
    ok = wait_mma(bar, phase, p.status, p.timeout_ns) && ok;
    phase ^= 1;
    ptx::tc_fence_after();
    if (warp < 4 && warp * 32 < m) {
      const int i = warp * 32 + lane;
      for (int c0 = 0; c0 < nmm; c0 += 32) {
        uint32_t r[32];
        ptx::tmem_ld_32x32b_x32(tmem + (static_cast<uint32_t>(warp * 32) << 16) + c0, r);
        ptx::tmem_ld_wait();
        if (i < m) {
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (c0 + j < m) sP[par * m * m + i * m + c0 + j] = __uint_as_float(r[j]);
        }
      }
    }
    ptx::tc_fence_before();
    ptx::cluster_sync();
    ptx::tc_fence_after();
    // A = sum of the partials in rank order (every CTA gets the same bits);
    // A stays fp32 here: it is never an MMA operand on this path.
    const float gscale = first ? inv * inv : 1.f;
    for (int e = tid; e < m * m; e += kSmallThreads) {
      const uint32_t a = ptx::smem_u32(sP + par * m * m + e);
      float v[kSmallMaxCluster];
#pragma unroll
      for (int r = 0; r < kSmallMaxCluster; ++r)
        v[r] = r < p.cs ? ptx::ld_shared_cluster_f32(ptx::mapa_shared(a, r)) : 0.f;
      float acc = 0.f;
#pragma unroll
      for (int r = 0; r < kSmallMaxCluster; ++r) acc += v[r];
      const int i = e / m, j = e - i * m;
      sA[i * (m + 1) + j] = acc * gscale;
    }
    __syncthreads();
    // P = a*I + b*A + c*A^2 in fp32, stored as two bf16 K-major operands
    // P = hi + lo (rows q < m, columns k < m): the apply multiplies by both,
    // so the bf16 rounding of P no longer limits the accuracy.
    for (int e = tid; e < m * m; e += kSmallThreads) {
      const int i = e / m, j = e - i * m;
      float s2 = 0.f;
      for (int k = 0; k < m; ++k) s2 = fmaf(sA[i * (m + 1) + k], sA[k * (m + 1) + j], s2);
      const float v = fmaf(cb, sA[i * (m + 1) + j], cc * s2) + (i == j ? ca + al : 0.f);
      const __nv_bfloat16 hi = __float2bfloat16_rn(v);
      const uint32_t off = ptx::sw128_offset(i, j * 2);
      *reinterpret_cast<__nv_bfloat16*>(sBt + off) = hi;
      *reinterpret_cast<__nv_bfloat16*>(sBt + kSmallBTile + off) =
          __float2bfloat16_rn(v - __bfloat162float(hi));
    }
    ptx::fence_proxy_async_smem();
    __syncthreads();
    // Apply, in batches of product tiles that fit the TMEM allocation
    const float xs = first ? inv : 1.f;
    for (int t0 = 0; t0 < tiles; t0 += per_batch) {
      const int nb = min(per_batch, tiles - t0);
      if (tid == 0) {
        ptx::tc_fence_after();
        for (int tt = 0; tt < nb; ++tt) {
          const int t = t0 + tt;
          for (int j = 0; j < nmm / 16; ++j) {
            const uint64_t a = ptx::sdesc_mnmajor_sw128(sX_u + 2 * t * chunk_bytes + j * 2048,
                                                        chunk_bytes, 1024);
            ptx::umma_bf16(tmem + tcol * (1 + tt), a, ptx::sdesc_kmajor_sw128(sBt_u + j * 32),
                           idesc_app, j != 0 ? 1u : 0u);
            ptx::umma_bf16(tmem + tcol * (1 + tt), a,
                           ptx::sdesc_kmajor_sw128(sBt_u + kSmallBTile + j * 32), idesc_app, 1u);
          }
        }
        ptx::umma_commit(bar);
      }
      __syncwarp();
      ok = wait_mma(bar, phase, p.status, p.timeout_ns) && ok;
      phase ^= 1;
      ptx::tc_fence_after();
      const int q4 = warp & 3;
      for (int tt = warp >> 2; tt < nb; tt += 2) {
        const int gp = 128 * (t0 + tt) + q4 * 32 + lane;       // X column within the CTA
        uint8_t* col = sX + (gp >> 6) * chunk_bytes;
        const uint32_t byte = (gp & 63) * 2;
        for (int c0 = 0; c0 < nmm; c0 += 32) {
          uint32_t r[32];
          ptx::tmem_ld_32x32b_x32(
              tmem + (static_cast<uint32_t>(q4 * 32) << 16) + tcol * (1 + tt) + c0, r);
          ptx::tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) {
            const int q = c0 + j;
            if (q < m)
              *reinterpret_cast<__nv_bfloat16*>(col + ptx::sw128_offset(q, byte)) =
                  __float2bfloat16_rn(xs * __uint_as_float(r[j]));
          }
        }
      }
      ptx::fence_proxy_async_smem();
      ptx::tc_fence_before();
      __syncthreads();
      ptx::tc_fence_after();
    }
  }

  // ---- update (or copy-back) from the cluster-resident result -----------------------
  const float os = p.steps == 0 ? inv : 1.f;
  const float decay = 1.f - p.lr * p.wd, stepk = p.lr * S.scale * os;
  if (ok) {
    for (int base = tid; base < items; base += kSmallUnroll * kSmallThreads) {
      float wv[kSmallUnroll][8];
      int64_t e[kSmallUnroll];
      int nv[kSmallUnroll], row[kSmallUnroll], jl[kSmallUnroll];
#pragma unroll
      for (int u = 0; u < kSmallUnroll; ++u) {
        const int item = base + u * kSmallThreads;
        nv[u] = 0;
        if (item < items) {
          if (!S.trans) {
            const int gpr = w / 8;
            row[u] = item / gpr;
            jl[u] = (item - row[u] * gpr) * 8;
            const int64_t gj = col0 + jl[u];
            if (gj < n) {
              nv[u] = (n - gj) < 8 ? static_cast<int>(n - gj) : 8;
              e[u] = moff + static_cast<int64_t>(row[u]) * n + gj;
            }
          } else {
            jl[u] = item / ig;
            row[u] = (item - jl[u] * ig) * 8;
            const int64_t gj = col0 + jl[u];
            if (gj < n) {
              nv[u] = min(8, m - row[u]);
              e[u] = moff + gj * m + row[u];
            }
          }
        }
        if (nv[u] > 0 && p.step_mode) load8(S.W, S.w_dtype, e[u], nv[u], S.wvec, wv[u]);
      }
#pragma unroll
      for (int u = 0; u < kSmallUnroll; ++u) {
        if (nv[u] <= 0) continue;
        const uint8_t* col = sX + (jl[u] >> 6) * chunk_bytes;
        const uint32_t byte = (jl[u] & 63) * 2;
        float o[8];
        if (!S.trans) {
          const uint4 q = *reinterpret_cast<const uint4*>(col + ptx::sw128_offset(row[u], byte));
          const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&q);
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const float2 f = __bfloat1622float2(h[j]);
            o[2 * j] = f.x;
            o[2 * j + 1] = f.y;
          }
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j)
            o[j] = j < nv[u] ? __bfloat162float(*reinterpret_cast<const __nv_bfloat16*>(
                                   col + ptx::sw128_offset(row[u] + j, byte)))
                             : 0.f;
        }
        if (p.step_mode) {
#pragma unroll
          for (int j = 0; j < 8; ++j) wv[u][j] = fmaf(decay, wv[u][j], -stepk * o[j]);
        } else {
#pragma unroll
          for (int j = 0; j < 8; ++j) wv[u][j] = o[j] * os;
        }
        store8(S.W, S.w_dtype, e[u], nv[u], S.wvec, wv[u]);
      }
    }
  }
  // No CTA leaves while a peer may still read its shared memory.
  ptx::tc_fence_before();
  ptx::cluster_sync();
  if (warp == 0) ptx::tmem_dealloc(tmem, kSmallTmemCols);
}

int small_max_active_clusters(int cs, int smem_bytes) {
  if (cudaFuncSetAttribute(ns_small_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           smem_bytes) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(cs), 1, 1);
  cfg.blockDim = dim3(kSmallThreads, 1, 1);
  cfg.dynamicSmemBytes = smem_bytes;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, ns_small_kernel, &cfg) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  return n;
}

cudaError_t launch_small(const SmallParams& p, int total_mats, cudaStream_t s) {
  if (total_mats <= 0) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(ns_small_kernel,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize, p.smem_bytes);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(total_mats) * p.cs, 1, 1);
  cfg.blockDim = dim3(kSmallThreads, 1, 1);
  cfg.dynamicSmemBytes = p.smem_bytes;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = p.cs;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, ns_small_kernel, p);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace muon
