// Allocation-free variant of the batched Newton-Schulz entry point.
//
// Some callers cannot call cudaMalloc: code that runs while an allocator is
// frozen or owned by someone else (a custom caching allocator that must see
// every device allocation, a host process with a fixed memory budget carved
// up in advance, a plugin loaded into a framework that forbids allocating
// outside its own pool).  For them this file keeps the whole workspace of one
// call in a fixed file-scope device array, so the call allocates nothing.
//
// Cost: every GPU that loads this library holds kScratchBytes of device memory
// until the process exits, whether or not the entry point is used.
//
// The host cannot use g_scratch's name as a device address; its address is
// taken once per device with cudaGetSymbolAddress (with that device current)
// on the first call made on that device.
#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>

#include "../../include/muon.h"
#include "muon_internal.h"

using namespace muon;

namespace {

constexpr size_t kScratchBytes = size_t(64) << 20;   // 64 MiB per device
constexpr int kMaxDevices = 64;
constexpr float kShiftFrac = 0.58f;
constexpr float kEps = 1e-7f;

__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_mu;
char* g_base[kMaxDevices];
int g_sms[kMaxDevices];

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

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t align_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

bool make_map(CUtensorMap* map, const void* base, int64_t inner, int64_t rows, int64_t cnt,
              int64_t pitch, int64_t mstride, int box_rows) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows),
                        static_cast<cuuint64_t>(cnt)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(pitch * 2),
                           static_cast<cuuint64_t>(mstride * 2)};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(gemm_block_k()),
                       static_cast<cuuint32_t>(box_rows), 1};
  cuuint32_t estr[3] = {1, 1, 1};
  return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
            box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) ==
         CUDA_SUCCESS;
}

// Set-up once per device (that device current): the device address of the
// scratch array and the SM count.
muon_status_t scratch_base(char** base, int* sms) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_CUDA;
  if (dev < 0 || dev >= kMaxDevices) return MUON_ERR_UNSUPPORTED;
  std::lock_guard<std::mutex> lock(g_mu);
  if (!g_base[dev]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) {
      cudaGetLastError();
      return MUON_ERR_CUDA;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MUON_ERR_CUDA;
    g_sms[dev] = n;
    g_base[dev] = static_cast<char*>(p);
  }
  *base = g_base[dev];
  *sms = g_sms[dev];
  return MUON_OK;
}

}  // namespace

extern "C" muon_status_t muon_ns_batched_noalloc(void* X, int64_t B, int64_t M, int64_t N,
                                                 int steps, float a, float b, float c,
                                                 cudaStream_t stream) {
  if (B < 0 || M < 0 || N < 0 || steps < 0 || steps > kMaxSteps) return MUON_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(a) || !std::isfinite(b) || !std::isfinite(c))
    return MUON_ERR_INVALID_ARGUMENT;
  if (B == 0 || M == 0 || N == 0) return MUON_OK;
  if (!X || (reinterpret_cast<uintptr_t>(X) & 1)) return MUON_ERR_INVALID_ARGUMENT;
  if (M > (1LL << 30) || N > (1LL << 30) || B > (1LL << 30)) return MUON_ERR_UNSUPPORTED;

  const bool trans = M > N;
  const int64_t m = trans ? N : M, n = trans ? M : N;
  const int bm = gemm_block_m(), bn = gemm_block_n(), bk = gemm_block_k();
  const int64_t m_pad = cdiv(m, 8) * 8, n_pad = cdiv(n, 8) * 8;
  const int64_t tri = gemm_sym_tiles(static_cast<int>(m));
  const int num_kb = static_cast<int>(cdiv(n, bk));
  const int64_t prep_tiles = cdiv(m, kPrepTile) * cdiv(n, kPrepTile);

  // Layout: [status | counters] (cleared every call) then the data buffers.
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + (bytes < 16 ? 16 : bytes), 256);
    return o;
  };
  const size_t o_status = take(sizeof(unsigned));
  const size_t o_cnt = take(static_cast<size_t>(B) * 4);
  const size_t o_tcnt = take(static_cast<size_t>(B * tri) * 4);
  const size_t zero_bytes = off;
  off = align_up(off, 1024);
  const size_t o_X = take(static_cast<size_t>(B * m * n_pad) * 2);
  const size_t o_Xt0 = take(static_cast<size_t>(B * n * m_pad) * 2);
  const size_t o_Xt1 = take(static_cast<size_t>(B * n * m_pad) * 2);
  const size_t o_A = take(static_cast<size_t>(B * m * m_pad) * 2);
  const size_t o_B = take(static_cast<size_t>(B * m * m_pad) * 2);
  const size_t o_inv = take(static_cast<size_t>(B) * 4);
  const size_t o_ssq = take(static_cast<size_t>(B * prep_tiles) * 4);
  // split-K heuristic of the allocating path, so both give the same bits
  char* base = nullptr;
  int sms = 0;
  muon_status_t st = scratch_base(&base, &sms);
  if (st != MUON_OK) return st;
  const int64_t gram_tiles = B * tri, target = 2LL * sms;
  int ks = 1;
  if (gram_tiles < target && num_kb >= 8) {
    ks = static_cast<int>(std::min<int64_t>(cdiv(target, gram_tiles), num_kb / 4));
    ks = ks < 1 ? 1 : ks;
  }
  const int kb_per_split = static_cast<int>(cdiv(num_kb, ks));
  const int ksplit = static_cast<int>(cdiv(num_kb, kb_per_split));
  const size_t o_part = take(ksplit > 1 ? static_cast<size_t>(B * tri * ksplit) * bm * bn * 4 : 16);
  if (off > kScratchBytes) return MUON_ERR_UNSUPPORTED;   // beyond the fixed scratch size
  const int64_t prep_blocks = B * cdiv(M, kPrepTile) * cdiv(N, kPrepTile);
  const int64_t fin_blocks = B * cdiv(M, kFinRows) * cdiv(N, kFinCols);
  if (prep_blocks >= (1LL << 31) || fin_blocks >= (1LL << 31)) return MUON_ERR_UNSUPPORTED;

  unsigned* status = reinterpret_cast<unsigned*>(base + o_status);
  unsigned* cnt = reinterpret_cast<unsigned*>(base + o_cnt);
  unsigned* tcnt = reinterpret_cast<unsigned*>(base + o_tcnt);
  auto* Xb = reinterpret_cast<__nv_bfloat16*>(base + o_X);
  __nv_bfloat16* Xt[2] = {reinterpret_cast<__nv_bfloat16*>(base + o_Xt0),
                          reinterpret_cast<__nv_bfloat16*>(base + o_Xt1)};
  auto* Ab = reinterpret_cast<__nv_bfloat16*>(base + o_A);
  auto* Bb = reinterpret_cast<__nv_bfloat16*>(base + o_B);
  float* inv = reinterpret_cast<float*>(base + o_inv);

  // The array keeps the previous call's contents: clear status and counters.
  if (cudaMemsetAsync(base, 0, zero_bytes, stream) != cudaSuccess) return MUON_ERR_CUDA;

  CUtensorMap mX, mXq, mA, mAq, mB, mXt[2];
  if (!make_map(&mX, Xb, n, m, B, n_pad, m * n_pad, bm) ||
      !make_map(&mXq, Xb, n, m, B, n_pad, m * n_pad, bn) ||
      !make_map(&mA, Ab, m, m, B, m_pad, m * m_pad, bm) ||
      !make_map(&mAq, Ab, m, m, B, m_pad, m * m_pad, bn) ||
      !make_map(&mB, Bb, m, m, B, m_pad, m * m_pad, bn) ||
      !make_map(&mXt[0], Xt[0], m, n, B, m_pad, n * m_pad, bm) ||
      !make_map(&mXt[1], Xt[1], m, n, B, m_pad, n * m_pad, bm))
    return MUON_ERR_CUDA;

  unsigned long long timeout_ns = 2000ull * 1000000ull;
  if (const char* v = std::getenv("MUON_WAIT_TIMEOUT_MS")) {
    const unsigned long long x = std::strtoull(v, nullptr, 10);
    if (x > 0) timeout_ns = x * 1000000ull;
  }

  // ---- prep: X0 = bf16(X) in both layouts and per-matrix 1/(||X||+eps) ----
  {
    PrepParams pp;
    std::memset(&pp, 0, sizeof(pp));
    PrepSlice& ps = pp.s[0];
    ps.G = X;
    ps.direct = trans ? Xt[0] : Xb;
    ps.transp = trans ? Xb : Xt[0];
    ps.pitch_d = trans ? m_pad : n_pad;
    ps.pitch_t = trans ? n_pad : m_pad;
    ps.mstride_d = trans ? n * m_pad : m * n_pad;
    ps.mstride_t = trans ? m * n_pad : n * m_pad;
    ps.ssq_part = reinterpret_cast<float*>(base + o_ssq);
    ps.inv = inv;
    ps.cnt = cnt;
    ps.r = M;
    ps.c = N;
    ps.count = static_cast<int>(B);
    ps.g_dtype = MUON_BF16;
    ps.tiles_r = static_cast<int>(cdiv(M, kPrepTile));
    ps.tiles_c = static_cast<int>(cdiv(N, kPrepTile));
    ps.tile_base = 0;
    ps.vec = (N % 8 == 0) && (reinterpret_cast<uintptr_t>(X) % 16 == 0);
    ps.trans = trans ? 1 : 0;
    pp.n_slices = 1;
    pp.total_blocks = static_cast<int>(prep_blocks);
    pp.step_mode = 0;
    pp.eps = kEps;
    pp.status = status;
    if (launch_prep(pp, stream) != cudaSuccess) return MUON_ERR_CUDA;
  }
  // ---- NS iterations ----
  for (int it = 0; it < steps; ++it) {
    for (int phase = 0; phase < 3; ++phase) {
      GemmParams gp;
      std::memset(&gp, 0, sizeof(gp));
      GemmGroup& G = gp.g[0];
      G.m = static_cast<int>(m);
      G.n = static_cast<int>(n);
      G.count = static_cast<int>(B);
      G.inv = inv;
      G.tile_base = 0;
      if (phase == kEpiGram) {
        G.mapA = mX;
        G.mapB = mXq;
        G.out0 = Ab;
        G.pitch0 = m_pad;
        G.mstride0 = m * m_pad;
        G.partial = reinterpret_cast<float*>(base + o_part);
        G.tile_cnt = tcnt;
        G.nt = static_cast<int>(cdiv(m, bn));
        G.mt = static_cast<int>(cdiv(m, bm));
        G.ksplit = ksplit;
        G.kb_per_split = kb_per_split;
        G.num_kb = num_kb;
        G.tiles_per_mat = static_cast<int>(tri * ksplit);
      } else if (phase == kEpiPoly) {
        G.mapA = mA;
        G.mapB = mAq;
        G.epi_in = Ab;
        G.pitch_in = m_pad;
        G.mstride_in = m * m_pad;
        G.out0 = Bb;
        G.pitch0 = m_pad;
        G.mstride0 = m * m_pad;
        G.nt = static_cast<int>(cdiv(m, bn));
        G.mt = static_cast<int>(cdiv(m, bm));
        G.ksplit = 1;
        G.num_kb = static_cast<int>(cdiv(m, bk));
        G.kb_per_split = G.num_kb;
        G.tiles_per_mat = static_cast<int>(tri);
      } else {
        G.mapA = mXt[it & 1];
        G.mapB = mB;
        G.epi_in = Xt[it & 1];
        G.pitch_in = m_pad;
        G.mstride_in = n * m_pad;
        G.out0 = Xt[(it + 1) & 1];
        G.pitch0 = m_pad;
        G.mstride0 = n * m_pad;
        G.out1 = Xb;
        G.pitch1 = n_pad;
        G.mstride1 = m * n_pad;
        G.nt = static_cast<int>(cdiv(m, bn));
        G.mt = static_cast<int>(cdiv(n, bm));
        G.ksplit = 1;
        G.num_kb = static_cast<int>(cdiv(m, bk));
        G.kb_per_split = G.num_kb;
        G.tiles_per_mat = G.nt * G.mt;
      }
      const int64_t tiles = static_cast<int64_t>(G.tiles_per_mat) * B;
      if (tiles >= (1LL << 31)) return MUON_ERR_UNSUPPORTED;
      gp.n_groups = 1;
      gp.total_tiles = static_cast<int>(tiles);
      const float alpha = kShiftFrac * a;
      gp.a = a - alpha;
      gp.b = b;
      gp.c = c;
      gp.alpha = alpha;
      gp.first = it == 0 ? 1 : 0;
      gp.status = status;
      gp.timeout_ns = timeout_ns;
      if (launch_gemm(phase, gp, stream) != cudaSuccess) return MUON_ERR_CUDA;
    }
  }
  // ---- copy-back into X ([M][N] layout) ----
  {
    FinParams fp;
    std::memset(&fp, 0, sizeof(fp));
    FinSlice& fs = fp.s[0];
    fs.W = X;
    const int fin = steps & 1;
    fs.O = trans ? Xt[fin] : Xb;
    fs.pitch_o = trans ? m_pad : n_pad;
    fs.mstride_o = trans ? n * m_pad : m * n_pad;
    fs.inv = steps == 0 ? inv : nullptr;
    fs.r = M;
    fs.c = N;
    fs.count = static_cast<int>(B);
    fs.w_dtype = MUON_BF16;
    fs.tiles_r = static_cast<int>(cdiv(M, kFinRows));
    fs.tiles_c = static_cast<int>(cdiv(N, kFinCols));
    fs.tile_base = 0;
    fs.vec = (N % 8 == 0) && (reinterpret_cast<uintptr_t>(X) % 16 == 0);
    fs.scale = 1.f;
    fp.n_slices = 1;
    fp.total_blocks = static_cast<int>(fin_blocks);
    fp.step_mode = 0;
    if (launch_finish(fp, stream) != cudaSuccess) return MUON_ERR_CUDA;
  }
  return MUON_OK;
}
