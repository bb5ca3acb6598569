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
//
// The array starts with a status word (device-detected conditions: a
// non-finite norm, a bounded wait that gave up).  It is cleared by the first
// call on a device and by muon_query_status, which reads it; every other
// call leaves it alone, so a condition stays visible until it is read.
// Behind it come the per-call counters (cleared by every call) and the data
// buffers of the grouped GEMM path.
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
bool g_status_clean[kMaxDevices];   // the first call on the device cleared the status word

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
size_t align_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

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

namespace muon {
unsigned* noalloc_status_word(int dev) {
  if (dev < 0 || dev >= kMaxDevices) return nullptr;
  std::lock_guard<std::mutex> lock(g_mu);
  return g_status_clean[dev] ? reinterpret_cast<unsigned*>(g_base[dev]) : nullptr;
}
}  // namespace muon

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
  const int64_t m_pad = cdiv(m, 8) * 8;
  const int64_t tri = gemm_sym_tiles(static_cast<int>(m));
  const int num_kb = static_cast<int>(cdiv(n, bk));
  const int64_t prep_tiles = cdiv(m, kPrepTile) * cdiv(n, kPrepTile);

  // Layout: status word, counters (cleared every call), data buffers.
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + (bytes < 16 ? 16 : bytes), 256);
    return o;
  };
  const size_t o_status = take(sizeof(unsigned));
  const size_t o_cnt = take(static_cast<size_t>(B) * 4);
  const size_t o_tcnt = take(static_cast<size_t>(B * tri) * 4);
  const size_t zero_end = off;
  off = align_up(off, 1024);
  const size_t o_Xt0 = take(static_cast<size_t>(B * n * m_pad) * 2);
  const size_t o_Xt1 = take(static_cast<size_t>(B * n * m_pad) * 2);
  const size_t o_A = take(static_cast<size_t>(B * m * m_pad) * 2);
  const size_t o_B = take(static_cast<size_t>(B * m * m_pad) * 2);
  const size_t o_inv = take(static_cast<size_t>(B) * 4);
  const size_t o_ssq = take(static_cast<size_t>(B * prep_tiles) * 4);
  // The split-K rule of the allocating path's grouped GEMMs (its cap
  // included).  The results agree with muon_ns_batched within the NS
  // tolerance, not bit for bit: that call also cuts large batches into
  // chunks and sends core shapes with min(M, N) <= 64 to its Gram-space
  // kernel, while this one runs every shape on the grouped GEMM path.
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
  {
    int cap = 64;
    if (const char* v = std::getenv("MUON_MAX_KSPLIT")) {
      const long x = std::strtol(v, nullptr, 10);
      if (x > 0) cap = static_cast<int>(std::min<long>(x, 1 << 20));
    }
    ks = std::min(ks, cap);
  }
  const int kb_per_split = static_cast<int>(cdiv(num_kb, ks));
  const int ksplit = static_cast<int>(cdiv(num_kb, kb_per_split));
  const size_t o_part = take(ksplit > 1 ? static_cast<size_t>(B * tri * ksplit) * bm * bn * 4 : 16);
  if (off > kScratchBytes) return MUON_ERR_UNSUPPORTED;   // beyond the fixed scratch size
  const int64_t prep_blocks = B * cdiv(M, kPrepTile) * cdiv(N, kPrepTile);
  const int64_t fin_blocks = trans ? B * cdiv(M, kFinRows) * cdiv(N, kFinCols)
                                   : B * cdiv(M, kFinTRows) * cdiv(N, kFinTCols);
  if (prep_blocks >= (1LL << 31) || fin_blocks >= (1LL << 31)) return MUON_ERR_UNSUPPORTED;

  unsigned* status = reinterpret_cast<unsigned*>(base + o_status);
  unsigned* cnt = reinterpret_cast<unsigned*>(base + o_cnt);
  unsigned* tcnt = reinterpret_cast<unsigned*>(base + o_tcnt);
  float* inv = reinterpret_cast<float*>(base + o_inv);
  NsGroupDev g;
  g.m = m;
  g.n = n;
  g.cnt = B;
  g.m_pad = m_pad;
  g.Xt[0] = reinterpret_cast<__nv_bfloat16*>(base + o_Xt0);
  g.Xt[1] = reinterpret_cast<__nv_bfloat16*>(base + o_Xt1);
  g.A = reinterpret_cast<__nv_bfloat16*>(base + o_A);
  g.B = reinterpret_cast<__nv_bfloat16*>(base + o_B);
  g.inv = inv;
  g.partial = reinterpret_cast<float*>(base + o_part);
  g.tile_cnt = tcnt;
  g.ksplit = ksplit;
  g.kb_per_split = kb_per_split;
  g.num_kb_gram = num_kb;
  g.tri = tri;

  // The array keeps the previous call's contents: clear the counters (and,
  // on the device's first call, the status word as well).
  {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_mu);
    const size_t from = g_status_clean[dev] ? o_cnt : o_status;
    if (cudaMemsetAsync(base + from, 0, zero_end - from, stream) != cudaSuccess) return MUON_ERR_CUDA;
    g_status_clean[dev] = true;
  }

  if (!ns_group_maps(g)) return MUON_ERR_CUDA;

  unsigned long long timeout_ns = 2000ull * 1000000ull;
  if (const char* v = std::getenv("MUON_WAIT_TIMEOUT_MS")) {
    const unsigned long long x = std::strtoull(v, nullptr, 10);
    if (x > 0) timeout_ns = x * 1000000ull;
  }

  // ---- prep: Xt = bf16(X0)^T-layout and per-matrix 1/(||X||+eps) ----
  {
    PrepParams pp;
    std::memset(&pp, 0, sizeof(pp));
    PrepSlice& ps = pp.s[0];
    ps.G = X;
    ps.direct = trans ? g.Xt[0] : nullptr;
    ps.transp = trans ? nullptr : g.Xt[0];
    ps.pitch_d = ps.pitch_t = m_pad;
    ps.mstride_d = ps.mstride_t = n * m_pad;
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
      ns_fill_group(G, g, phase, it, 0);
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
      gp.deep = gemm_deep(phase, G.kb_per_split);
      gp.status = status;
      gp.timeout_ns = timeout_ns;
      gp.inject = take_injected_stall(kInjectGemm);
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
    fs.O = g.Xt[fin];
    fs.o_trans = trans ? 0 : 1;
    fs.pitch_o = m_pad;
    fs.mstride_o = n * m_pad;
    fs.inv = steps == 0 ? inv : nullptr;
    fs.r = M;
    fs.c = N;
    fs.count = static_cast<int>(B);
    fs.w_dtype = MUON_BF16;
    fs.tiles_r = static_cast<int>(cdiv(M, fs.o_trans ? kFinTRows : kFinRows));
    fs.tiles_c = static_cast<int>(cdiv(N, fs.o_trans ? kFinTCols : kFinCols));
    fs.tile_base = 0;
    fs.vec = (N % 8 == 0) && (reinterpret_cast<uintptr_t>(X) % 16 == 0);
    fs.scale = 1.f;
    fp.n_slices = 1;
    fp.total_blocks = static_cast<int>(fin_blocks);
    fp.status = status;
    fp.step_mode = 0;
    if (launch_finish(fp, stream) != cudaSuccess) return MUON_ERR_CUDA;
  }
  return MUON_OK;
}
