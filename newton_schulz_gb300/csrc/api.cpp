// C ABI of libmuon: argument validation, the core-shape planner, the
// workspace cache, tensor-map construction and kernel launches.
//
// Planner (HyperParallel-FSDP section 6.6, Fig. 10(a)): every slice of every
// group becomes one NS problem with m = min(rows, cols), n = max(rows, cols)
// (transpose-first when rows > cols); problems with the same core shape
// (m, n) share one workspace region and one set of tensor maps, so a single
// launch per phase covers all of them.  Work is cut into chunks whose X
// operands hold at most `cap` elements (2^29 by default, the page's
// memory-safe batch cap; MUON_WS_CAP overrides); one workspace, sized for the
// largest chunk, is allocated once per (device, stream) and reused.
#include <algorithm>
#include <atomic>
#include <cstdint>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <utility>
#include <vector>

#include "../../include/muon.h"
#include "muon_internal.h"

using namespace muon;

namespace {

constexpr float kDefA = 3.4445f, kDefB = -4.7750f, kDefC = 2.0315f, kDefEps = 1e-7f;
constexpr int kDefSteps = 5;
constexpr float kShiftFrac = 0.58f;   // alpha_k = 0.58 a_k (about 2 for the default quintic)

// ---- global state ---------------------------------------------------------------
// Data workspace (operands, Gram/polynomial buffers, partials) plus a
// separate counter buffer.  Every kernel leaves the counters it uses at zero,
// and counters never share memory with data, so a new plan (other offsets)
// always starts from zeroed counters.
struct Workspace {
  void* ptr = nullptr;
  size_t bytes = 0;
  unsigned* ctr = nullptr;
  size_t ctr_bytes = 0;
  bool dirty = false;  // a kernel gave up mid-way: counters must be re-zeroed
  // small-m path: per-matrix arrival counters and ready flags, tagged with a
  // launch epoch (never reset; a fresh allocation is zero = no epoch)
  unsigned long long* ep = nullptr;
  size_t ep_cap = 0;   // matrices
  unsigned epoch = 0;
};

struct DevState {
  unsigned* status = nullptr;
  int sms = 0;
  unsigned long long* guard_bad = nullptr;   // guard mode: bytes found changed in the bands
};

struct ProfRec {
  int kind;
  cudaEvent_t e0, e1;
};

std::mutex g_mu;
std::map<std::pair<int, cudaStream_t>, Workspace> g_ws;

// Host-resident steps (muon_step_grouped_host): per (device, caller stream),
// the copy-in, compute and copy-out streams, slot events and the device
// slots the chunks are staged through.
constexpr int kHostSlots = 3;
struct HostPipe {
  cudaStream_t s_in = nullptr, s_comp = nullptr, s_out = nullptr;
  cudaEvent_t ev_start = nullptr, ev_in[kHostSlots] = {}, ev_comp[kHostSlots] = {},
              ev_free[kHostSlots] = {};
  void* slot = nullptr;   // kHostSlots x slot_bytes
  size_t slot_bytes = 0;
};
std::map<std::pair<int, cudaStream_t>, HostPipe> g_host;
std::map<int, DevState> g_dev;
std::atomic<int> g_inject{0};   // muon_debug_inject_stall: one pending request
bool g_prof = false;
std::vector<ProfRec> g_prof_recs;
thread_local int t_last_launches = 0;

size_t env_size(const char* name, size_t dflt) {
  const char* v = std::getenv(name);
  if (!v || !*v) return dflt;
  char* end = nullptr;
  unsigned long long x = std::strtoull(v, &end, 10);
  return (end && *end == 0 && x > 0) ? static_cast<size_t>(x) : dflt;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }
int64_t rup(int64_t a, int64_t b) { return cdiv(a, b) * b; }
size_t align_up(size_t a, size_t b) { return (a + b - 1) / b * b; }

muon_status_t dev_state(DevState** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_CUDA;
  DevState& d = g_dev[dev];
  if (!d.status) {
    if (cudaMalloc(&d.status, 256) != cudaSuccess) {
      d.status = nullptr;
      return MUON_ERR_OUT_OF_MEMORY;
    }
    if (cudaMemset(d.status, 0, 256) != cudaSuccess) return MUON_ERR_CUDA;
    if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return MUON_ERR_CUDA;
  }
  *out = &d;
  return MUON_OK;
}

// ---- guard mode --------------------------------------------------------------------
// Guard mode (MUON_WS_GUARD=1, a debugging aid): every workspace buffer is
// followed by a band of kGuardBytes that no kernel may write; the bands are
// filled with kGuardByte before a layout's launches and counted by
// guard_check_kernel after them (read with muon_debug_guard_check).
constexpr size_t kGuardBytes = 4096;
constexpr int kGuardByte = 0xA5;
muon_status_t guard_counter(DevState* dev) {
  if (dev->guard_bad) return MUON_OK;
  if (cudaMalloc(&dev->guard_bad, sizeof(unsigned long long)) != cudaSuccess) {
    cudaGetLastError();
    dev->guard_bad = nullptr;
    return MUON_ERR_OUT_OF_MEMORY;
  }
  return cudaMemset(dev->guard_bad, 0, sizeof(unsigned long long)) == cudaSuccess ? MUON_OK
                                                                                    : MUON_ERR_CUDA;
}

muon_status_t guard_fill(char* ws, const std::vector<size_t>& bands, size_t bytes,
                         cudaStream_t stream) {
  for (size_t o : bands)
    if (cudaMemsetAsync(ws + o, kGuardByte, bytes, stream) != cudaSuccess) return MUON_ERR_CUDA;
  return MUON_OK;
}

muon_status_t guard_check(char* ws, const std::vector<size_t>& bands, size_t bytes,
                          DevState* dev, cudaStream_t stream) {
  for (size_t b = 0; b < bands.size(); b += kGuardMaxBands) {
    GuardParams gp;
    std::memset(&gp, 0, sizeof(gp));
    gp.base = reinterpret_cast<const uint8_t*>(ws);
    gp.n = static_cast<int>(std::min<size_t>(kGuardMaxBands, bands.size() - b));
    for (int i = 0; i < gp.n; ++i) gp.off[i] = bands[b + i];
    gp.bytes = static_cast<unsigned>(bytes);
    gp.pattern = static_cast<unsigned>(kGuardByte);
    gp.bad = dev->guard_bad;
    if (launch_guard_check(gp, stream) != cudaSuccess) return MUON_ERR_CUDA;
  }
  return MUON_OK;
}

// ---- plan --------------------------------------------------------------------------
struct Req {            // one user group
  void* W;
  int w_dtype;
  const void* G;
  int g_dtype;
  float* Mom;
  int64_t B, r, c, m, n;
  bool trans;
  bool gs = false;      // grouped GEMM path in Gram space (see gram_space_shape)
};

struct SliceP {
  int req;
  int64_t b0, cnt;
  int ng;
  int64_t idx0;
};

struct NsGroupP {
  int64_t m, n, cnt = 0;
  int64_t m_pad;
  int ksplit = 1, kb_per_split = 1, num_kb_gram = 1;
  int64_t tri = 1, prep_tiles = 1;
  size_t off_Xt0, off_Xt1, off_A, off_B, off_inv, off_ssq, off_part;
  size_t off_lo = 0;           // high-precision mode: Xt0, Xt1, A, B lo halves from here
  size_t off_S[5] = {0, 0, 0, 0, 0};   // Gram space: R, T, B', Q ping-pong (m x m_pad)
  size_t ctr_prep, ctr_tile;   // element offsets in the counter buffer
};

struct ChunkP {
  bool gs = false;             // every group of the chunk runs in Gram space
  std::vector<SliceP> slices;
  std::vector<NsGroupP> groups;
  size_t bytes = 0;
  size_t ctrs = 0;             // counters used (elements)
  std::vector<size_t> guards;  // guard-band offsets (MUON_WS_GUARD)
};

void layout_chunk(ChunkP& ch, int sms, bool precise, size_t guard) {
  size_t off = 0;
  auto take = [&](size_t bytes, bool band = true) {
    size_t o = off;
    off = align_up(off + std::max<size_t>(bytes, 16), 1024);
    if (guard && band) {
      ch.guards.push_back(off);
      off += guard;
    }
    return o;
  };
  const int bm = gemm_block_m(), bn = gemm_block_n(), bk = gemm_block_k();
  size_t ctr = 0;
  // split-K for the Gram only when the launch's symmetric tiles (all groups
  // together) cannot fill the GPU
  int64_t launch_tiles = 0;
  for (auto& g : ch.groups) launch_tiles += g.cnt * gemm_sym_tiles(static_cast<int>(g.m));
  for (auto& g : ch.groups) {
    g.m_pad = rup(g.m, 8);
    g.tri = gemm_sym_tiles(static_cast<int>(g.m));
    g.num_kb_gram = static_cast<int>(cdiv(g.n, bk));
    const int64_t tiles = launch_tiles;
    const int64_t target = 2LL * sms;
    int ks = 1;
    if (tiles < target && g.num_kb_gram >= 8) {
      ks = static_cast<int>(std::min<int64_t>(cdiv(target, std::max<int64_t>(tiles, 1)),
                                               g.num_kb_gram / 4));
      ks = std::max(ks, 1);
    }
    ks = std::min<int>(ks, static_cast<int>(env_size("MUON_MAX_KSPLIT", 64)));
    g.kb_per_split = static_cast<int>(cdiv(g.num_kb_gram, ks));
    g.ksplit = static_cast<int>(cdiv(g.num_kb_gram, g.kb_per_split));
    g.prep_tiles = cdiv(g.m, kPrepTile) * cdiv(g.n, kPrepTile);
    const size_t e2 = 2;
    g.off_Xt0 = take(static_cast<size_t>(g.cnt * g.n * g.m_pad) * e2);
    g.off_Xt1 = take(static_cast<size_t>(g.cnt * g.n * g.m_pad) * e2);
    if (ch.gs) {
      for (int i = 0; i < 5; ++i) g.off_S[i] = take(static_cast<size_t>(g.cnt * g.m * g.m_pad) * e2);
      g.off_A = g.off_S[kGsR];   // (the X-space maps are built on these, never used)
      g.off_B = g.off_S[kGsB];
    } else {
      g.off_A = take(static_cast<size_t>(g.cnt * g.m * g.m_pad) * e2);
      g.off_B = take(static_cast<size_t>(g.cnt * g.m * g.m_pad) * e2);
    }
    g.off_inv = take(static_cast<size_t>(g.cnt) * 4);
    g.off_ssq = take(static_cast<size_t>(g.cnt * g.prep_tiles) * 4);
    g.off_part = take(g.ksplit > 1 ? static_cast<size_t>(g.cnt * g.tri * g.ksplit) * bm * bn * 4
                                   : 16);
    if (precise) {   // lo halves, laid out like the hi ones (one band after all four)
      g.off_lo = take(static_cast<size_t>(g.cnt * g.n * g.m_pad) * e2, false);
      take(static_cast<size_t>(g.cnt * g.n * g.m_pad) * e2, false);
      take(static_cast<size_t>(g.cnt * g.m * g.m_pad) * e2, false);
      take(static_cast<size_t>(g.cnt * g.m * g.m_pad) * e2);
    }
    g.ctr_prep = ctr;
    ctr += static_cast<size_t>(g.cnt);
    g.ctr_tile = ctr;
    ctr += static_cast<size_t>(g.cnt * g.tri);
  }
  ch.bytes = off;
  ch.ctrs = ctr;
}

struct NsCfg {
  int steps;
  std::vector<float> coeffs;   // [steps][3]
  float eps;
  bool precise = false;        // MUON_NS_TF32: X0 carried as bf16 hi + lo
};

// Gram-space NS on the grouped GEMM path (DMuon-2 Appendix C.3), per core
// shape (m, n): with the symmetric m x m products on the polynomial kernel
// a matrix costs about (3 r + 18) m^3 algorithmic flops for r = n / m
// (Gram once, four symmetric products per step, one final apply) against
// (15 r + 5) m^3 in X space, so it is taken from r >= 2 on (bf16 products
// only; MUON_GRAM_SPACE=0 / 1 forbids / forces it, MUON_GRAM_SPACE_RATIO sets
// the r from which it is used).
// Gram-space restart period in NS steps for core shapes with small side m
// (MUON_GRAM_RESTART; 0: no restart).  Default: 3 for m >= 1024, else 2.
// Update error against the float64 oracle (one Gaussian matrix per shape,
// GB300): m = 768: P = 2 0.0087, P = 3 0.0110; m = 1024 ... 8192: P = 3
// 0.0062-0.0086, P = 2 0.0080-0.0121 (the 1e-2 ||dW|| bound).
int gram_restart_period_env(int64_t m) {
  const char* v = std::getenv("MUON_GRAM_RESTART");
  if (!v || !*v) return m >= 1024 ? 3 : 2;
  const long p = std::strtol(v, nullptr, 10);
  return p < 0 ? 2 : static_cast<int>(std::min<long>(p, 1 << 20));
}

int gram_restart_period(int64_t m) {
  const int p = gram_restart_period_env(m);
  return p == 0 ? (1 << 30) : p;
}

int gram_phases(int steps, int64_t m) {
  const int p = gram_restart_period(m);
  return steps <= 0 ? 0 : (steps + p - 1) / p;
}

// Gram space (the default iteration of DMuon-2 Appendix C.3) for core shapes
// with m >= 1024 and n >= ratio x m (MUON_GRAM_SPACE_RATIO, default 2) in
// bf16 mode: there its restart period is 3 and its update error measured
// 0.0062-0.0086 of ||dW|| against 0.0059-0.0069 in X space (the bound is
// 1e-2) for 9-24 % less time per step.  Below m = 1024 the period-2 form
// saved 1.3 % on the MoE experts (m = 768) at 0.0086 against 0.0072, and
// at m = 33 its NS error reached 0.031, so those shapes stay in X space.
// MUON_GRAM_SPACE=0 turns it off, =force applies it to every shape of the
// GEMM path.
constexpr int64_t kGramSpaceMinM = 1024;
bool gram_space_shape(int64_t m, int64_t n, const NsCfg& ns) {
  if (ns.precise || ns.steps < 1) return false;
  const char* v = std::getenv("MUON_GRAM_SPACE");
  if (v && std::strcmp(v, "force") == 0) return true;
  if (v && v[0] == '0') return false;
  const double ratio = static_cast<double>(env_size("MUON_GRAM_SPACE_RATIO", 2));
  return m >= kGramSpaceMinM && static_cast<double>(n) >= ratio * static_cast<double>(m);
}

// Row passes of an update launch: two (finish_tall_kernel: tiles twice as
// tall, 16 elements a thread) when every weight it writes is bf16 -- that
// kernel handles bf16 weights only -- else one.  MUON_FIN_PASSES=1 forces
// one pass.
int fin_passes(const std::vector<SliceP>& slices, const std::vector<Req>& reqs) {
  const char* v = std::getenv("MUON_FIN_PASSES");
  if (v && v[0] == '1') return 1;
  for (const SliceP& s : slices)
    if (reqs[s.req].w_dtype != MUON_BF16) return 1;
  return 2;
}

// Small-m path eligibility: core shapes with m <= 64 (MUON_SMALL_PATH=0 sends
// every shape to the grouped GEMM path).
bool small_shape(int64_t m) {
  const char* env = std::getenv("MUON_SMALL_PATH");
  if (env && env[0] == '0') return false;
  return m <= kSmallMaxM;
}

// Work items and shared-memory carve-up of the small-m kernel for core shape
// (m, n) over `mats` matrices; false when no carve-up fits one SM.  Shared
// memory holds a ring of stages, two Q images and the Gram-space matrices.
// A stage holds the data tile(s) of its phase (G + Mom: m x cw1, or W:
// m x 128, for the widest dtypes in the launch), then an X0 tile of 128
// columns at x_off and a 2 KB zero gap.  Items are up to 2560 columns (the
// X0 image of an item streams through the stages), shrinking while the
// launch would leave SMs without an item and a matrix keeps at most 10.
bool small_plan(int64_t m, int64_t n, int64_t mats, int sms, int esg, int esw, bool step,
                bool precise, SmallParams* sp) {
  sp->m = static_cast<int>(m);
  sp->n = static_cast<int>(n);
  sp->mr = static_cast<int>(rup(m, 8));
  sp->mp = m <= 32 ? 32 : 64;
  sp->nmm = static_cast<int>(rup(m, 16));
  sp->cw1 = m <= 32 ? 128 : 64;
  sp->qbytes = 2 * sp->nmm * 128;
  sp->pstride = static_cast<int>(rup(2 * m * m, 4));
  sp->precise = precise ? 1 : 0;
  sp->nblk = (sp->cw1 == 128 || precise) ? 2 : 1;
  sp->gcols = (precise && m > 32) ? 128 : 64;
  const size_t xs = precise ? 2 : 1;                          // X0 regions per 64 columns
  const size_t chunk = static_cast<size_t>(sp->mr) * 128;   // 64 X columns of X0
  const size_t p1 = static_cast<size_t>(m) * sp->cw1 * (esg + (step ? 4 : 0));
  const size_t p2 = static_cast<size_t>(m) * 128 * esw;
  sp->x_off = static_cast<int>(align_up(std::max(p1, p2), 1024));
  sp->stage_bytes = static_cast<int>(align_up(sp->x_off + 2 * xs * chunk + 2048, 1024));
  // the precise carve-up with 64 x 64 Gram-space matrices keeps three of them
  sp->gs_lowmem = (precise && sp->mp == 64) ? 1 : 0;
  const size_t gs =
      align_up(static_cast<size_t>(sp->gs_lowmem ? 3 : 5) * sp->mp * sp->mp * 4 + 64, 16);
  const size_t fixed = 2 * static_cast<size_t>(sp->qbytes) + gs + (kSmallCons / 32) * 512 + 512 + 1024;
  if (fixed >= static_cast<size_t>(kSmallSmemLimit)) return false;
  const int tcol = static_cast<int>(rup(sp->nmm, 32));
  // TMEM: two Gram accumulators in [0, 2 gcols), one O slot (2 tcol columns) per stage
  const int ocols = kSmallTmemCols - 2 * sp->gcols;
  sp->stages = static_cast<int>(std::min<size_t>((kSmallSmemLimit - fixed) / sp->stage_bytes,
                                                 std::min(kSmallMaxStages, ocols / (2 * tcol))));
  if (sp->stages < 2) return false;
  // items of at most 2560 columns (MUON_SMALL_ITEM_COLS; on 74 x [24, 10240]
  // items of 1280 / 2048 / 2560 / 3456 columns took 0.099 / 0.093 / 0.091 /
  // 0.096 ms)
  const int64_t cap =
      std::max<int64_t>(128, static_cast<int64_t>(env_size("MUON_SMALL_ITEM_COLS", 2560)));
  int64_t wb = std::min<int64_t>(cap, rup(n, 128));
  wb = rup(cdiv(n, cdiv(n, wb)), 128);
  {
    // Items shrink while the launch has fewer items than SMs, as long as a
    // matrix keeps at most 10 of them: each item adds a partial Gram that the
    // matrix's Gram-space job sums serially.  On [24, 10240] matrices,
    // 128-column items with two per SM took 208 / 137 / 86 us for 5 / 9 / 19
    // matrices, this rule 57 / 58 / 60 us; small n still splits (4 x [64, 256]
    // runs on 128-column items).
    const int64_t max_nb = static_cast<int64_t>(env_size("MUON_SMALL_MAX_ITEMS", 10));
    while (wb > 128 && mats * cdiv(n, wb) < static_cast<int64_t>(sms) &&
           cdiv(n, wb - 128) <= max_nb)
      wb -= 128;
  }
  sp->wb = static_cast<int>(wb);
  // second-phase claims: units of 2 tiles, up to 4 units per claim while
  // much work remains, 1 at the end (on 74 x [24, 10240] claims of a fixed
  // 16 / 8 / 4 / 2 tiles took 0.112 / 0.106 / 0.103 / 0.105 ms: large claims
  // spare the claim's round trips, small ones even out the end)
  sp->p2_tiles = std::max<int>(1, static_cast<int>(env_size("MUON_SMALL_P2_TILES", 2)));
  sp->p2_units = std::max<int>(1, static_cast<int>(env_size("MUON_SMALL_P2_UNITS", 4)));
  {
    const char* v = std::getenv("MUON_SMALL_TMA_STORE");
    sp->p2_tma_store = (v && v[0] == '0') ? 0 : 1;
  }
  sp->nb = static_cast<int>(cdiv(n, wb));
  sp->total_mats = static_cast<int>(mats);
  sp->items = static_cast<int>(mats * sp->nb);
  sp->xbytes = static_cast<int>((wb / 64) * xs * chunk);
  sp->off_ring = 0;
  sp->off_q = sp->stages * sp->stage_bytes;
  sp->off_gs = sp->off_q + 2 * sp->qbytes;
  sp->off_epi = static_cast<int>(align_up(sp->off_gs + gs, 16));
  sp->off_bar = sp->off_epi + (kSmallCons / 32) * 512;
  sp->smem_bytes = sp->off_bar + 512 + 1024;
  return sp->smem_bytes <= kSmallSmemLimit;
}

// Workspace of one small-m launch: X0 images, partial Grams, Q images (each
// followed by a guard band in guard mode); offsets into `off[3]`, guard-band
// offsets into `bands[3]`; returns the bytes.
size_t small_ws_layout(const SmallParams& sp, size_t guard, size_t* off, size_t* bands) {
  const size_t sizes[3] = {static_cast<size_t>(sp.items) * sp.xbytes,
                           static_cast<size_t>(sp.items) * sp.pstride * 4,
                           static_cast<size_t>(sp.total_mats) * sp.qbytes};
  size_t o = 0;
  for (int i = 0; i < 3; ++i) {
    off[i] = o;
    o = align_up(o + sizes[i], 256);
    bands[i] = o;
    o += guard;
  }
  return o;
}

std::vector<ChunkP> make_plan(const std::vector<Req>& reqs, int sms, bool precise, size_t guard) {
  const int64_t cap = static_cast<int64_t>(env_size("MUON_WS_CAP", size_t(1) << 29));
  std::vector<int> order;
  for (int i = 0; i < static_cast<int>(reqs.size()); ++i)
    if (reqs[i].B > 0 && reqs[i].m > 0) order.push_back(i);
  // largest matrices first; same core shapes adjacent
  std::stable_sort(order.begin(), order.end(), [&](int x, int y) {
    const Req &a = reqs[x], &b = reqs[y];
    if (a.m * a.n != b.m * b.n) return a.m * a.n > b.m * b.n;
    if (a.m != b.m) return a.m > b.m;
    return false;
  });
  std::vector<ChunkP> chunks;
  ChunkP cur;
  int64_t cur_elems = 0;
  auto close = [&] {
    const bool gs = cur.gs;
    if (!cur.slices.empty()) chunks.push_back(std::move(cur));
    cur = ChunkP();
    cur.gs = gs;
    cur_elems = 0;
  };
  for (int ri : order) {
    const Req& q = reqs[ri];
    const int64_t per = q.m * q.n;
    int64_t b = 0;
    // a chunk runs either in X space or in Gram space
    if (!cur.slices.empty() && cur.gs != q.gs) close();
    cur.gs = q.gs;
    while (b < q.B) {
      int ng = -1;
      for (int k = 0; k < static_cast<int>(cur.groups.size()); ++k)
        if (cur.groups[k].m == q.m && cur.groups[k].n == q.n) ng = k;
      const bool need_group = ng < 0;
      const bool full_tables = static_cast<int>(cur.slices.size()) >= kMaxSlices ||
                               (need_group && static_cast<int>(cur.groups.size()) >= kMaxNsGroups);
      int64_t fit = (cap - cur_elems) / per;
      if (!cur.slices.empty() && (fit <= 0 || full_tables)) {
        close();
        continue;
      }
      if (fit <= 0) fit = 1;   // one matrix larger than the cap runs alone
      const int64_t take = std::min(q.B - b, fit);
      if (need_group) {
        NsGroupP g;
        g.m = q.m;
        g.n = q.n;
        cur.groups.push_back(g);
        ng = static_cast<int>(cur.groups.size()) - 1;
      }
      SliceP s;
      s.req = ri;
      s.b0 = b;
      s.cnt = take;
      s.ng = ng;
      s.idx0 = cur.groups[ng].cnt;
      cur.groups[ng].cnt += take;
      cur.slices.push_back(s);
      cur_elems += take * per;
      b += take;
    }
  }
  close();
  for (auto& ch : chunks) layout_chunk(ch, sms, precise, guard);
  return chunks;
}

// ---- workspace ---------------------------------------------------------------------
muon_status_t get_workspace(cudaStream_t stream, size_t bytes, size_t ctrs, char** out,
                            unsigned** ctr_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_CUDA;
  Workspace& w = g_ws[{dev, stream}];
  const size_t ctr_bytes = std::max<size_t>(ctrs, 1) * sizeof(unsigned);
  if (w.bytes < bytes || w.ctr_bytes < ctr_bytes) {
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MUON_ERR_CUDA;
  }
  if (w.bytes < bytes) {
    if (w.ptr) cudaFree(w.ptr);
    w.ptr = nullptr;
    w.bytes = 0;
    const size_t want = align_up(bytes, size_t(1) << 21);
    if (cudaMalloc(&w.ptr, want) != cudaSuccess) {
      cudaGetLastError();
      w.ptr = nullptr;
      return MUON_ERR_OUT_OF_MEMORY;
    }
    w.bytes = want;
  }
  if (w.ctr_bytes < ctr_bytes) {
    if (w.ctr) cudaFree(w.ctr);
    w.ctr = nullptr;
    w.ctr_bytes = 0;
    const size_t want = align_up(ctr_bytes, size_t(1) << 16);
    if (cudaMalloc(&w.ctr, want) != cudaSuccess) {
      cudaGetLastError();
      w.ctr = nullptr;
      return MUON_ERR_OUT_OF_MEMORY;
    }
    w.ctr_bytes = want;
    w.dirty = true;
  }
  if (w.dirty) {
    if (cudaMemsetAsync(w.ctr, 0, w.ctr_bytes, stream) != cudaSuccess) return MUON_ERR_CUDA;
    w.dirty = false;
  }
  *out = static_cast<char*>(w.ptr);
  *ctr_out = w.ctr;
  return MUON_OK;
}

// Launch-tagged words of the small-m path for `mats` matrices: ready_list[cap]
// (epoch-tagged entries), the two arrive slots [2][cap] and the ring of
// per-launch counter slots; returns the next epoch (never 0) and cap.
muon_status_t get_epoch_ctrs(cudaStream_t stream, size_t mats, unsigned** arrive,
                             unsigned long long** ready_list, unsigned** ctr, unsigned* epoch,
                             int* cap_out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_CUDA;
  Workspace& w = g_ws[{dev, stream}];
  mats = std::max<size_t>(mats, 1);
  if (w.ep_cap < mats) {
    if (w.ep) {
      if (cudaStreamSynchronize(stream) != cudaSuccess) return MUON_ERR_CUDA;
      cudaFree(w.ep);
    }
    w.ep = nullptr;
    w.ep_cap = 0;
    const size_t cap = align_up(mats, 1024);
    const size_t bytes = cap * sizeof(unsigned long long) + 2 * cap * sizeof(unsigned) +
                         kSmallCtrSlots * 4 * sizeof(unsigned);
    if (cudaMalloc(&w.ep, bytes) != cudaSuccess) {
      cudaGetLastError();
      w.ep = nullptr;
      return MUON_ERR_OUT_OF_MEMORY;
    }
    if (cudaMemsetAsync(w.ep, 0, bytes, stream) != cudaSuccess) return MUON_ERR_CUDA;
    w.ep_cap = cap;
  }
  if (++w.epoch == 0) w.epoch = 1;
  *ready_list = w.ep;
  *arrive = reinterpret_cast<unsigned*>(w.ep + w.ep_cap);
  *ctr = *arrive + 2 * w.ep_cap;
  *cap_out = static_cast<int>(w.ep_cap);
  *epoch = w.epoch;
  return MUON_OK;
}

// ---- tensor maps ---------------------------------------------------------------------
// Tensor map of a stored [cnt][rows][inner] tensor for unswizzled tile copies
// of box {box_inner, box_rows, 1}; false when the layout is not TMA-legal.
bool make_tile_map(CUtensorMap* map, const void* base, int dtype, int64_t inner, int64_t rows,
                   int64_t cnt, int box_inner, int box_rows) {
  const int64_t es = dtype == MUON_F32 ? 4 : 2;
  const uint64_t dims[3] = {static_cast<uint64_t>(inner), static_cast<uint64_t>(rows),
                            static_cast<uint64_t>(cnt)};
  const uint64_t strides[2] = {static_cast<uint64_t>(inner * es),
                               static_cast<uint64_t>(inner * rows * es)};
  const uint32_t box[3] = {static_cast<uint32_t>(box_inner), static_cast<uint32_t>(box_rows), 1};
  return encode_tiled(map, dtype == MUON_F32, base, dims, strides, box, false);
}

// ---- launches ----------------------------------------------------------------------
struct Launcher {
  cudaStream_t stream;
  int count = 0;
  template <typename F>
  muon_status_t run(int kind, F&& f) {
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (g_prof) {
      cudaEventCreate(&e0);
      cudaEventCreate(&e1);
      cudaEventRecord(e0, stream);
    }
    cudaError_t e = f();
    if (e != cudaSuccess) {
      if (e0) cudaEventDestroy(e0);
      if (e1) cudaEventDestroy(e1);
      return MUON_ERR_CUDA;
    }
    if (g_prof) {
      cudaEventRecord(e1, stream);
      g_prof_recs.push_back({kind, e0, e1});
    }
    ++count;
    return MUON_OK;
  }
};


muon_status_t check_ns_cfg(const muon_ns_config_t* cfg, NsCfg* out) {
  if (!cfg) {
    out->steps = kDefSteps;
    out->coeffs.clear();
    for (int i = 0; i < kDefSteps; ++i) out->coeffs.insert(out->coeffs.end(), {kDefA, kDefB, kDefC});
    out->eps = kDefEps;
    return MUON_OK;
  }
  if (cfg->steps < 0 || cfg->steps > kMaxSteps) return MUON_ERR_INVALID_ARGUMENT;
  if (cfg->precision != MUON_NS_BF16 && cfg->precision != MUON_NS_TF32)
    return MUON_ERR_INVALID_ARGUMENT;
  out->precise = cfg->precision == MUON_NS_TF32;
  if (!std::isfinite(cfg->eps) || cfg->eps < 0.f) return MUON_ERR_INVALID_ARGUMENT;
  out->steps = cfg->steps;
  out->eps = cfg->eps;
  out->coeffs.clear();
  for (int i = 0; i < cfg->steps; ++i) {
    float a = cfg->a, b = cfg->b, c = cfg->c;
    if (cfg->coeffs) {
      a = cfg->coeffs[3 * i];
      b = cfg->coeffs[3 * i + 1];
      c = cfg->coeffs[3 * i + 2];
    }
    if (!std::isfinite(a) || !std::isfinite(b) || !std::isfinite(c))
      return MUON_ERR_INVALID_ARGUMENT;
    out->coeffs.insert(out->coeffs.end(), {a, b, c});
  }
  return MUON_OK;
}

float scale_value(int64_t r, int64_t c, int rule) {
  switch (rule) {
    case MUON_SCALE_SQRT_MAX1_R_OVER_C:
      return static_cast<float>(std::sqrt(std::max(1.0, double(r) / double(c))));
    case MUON_SCALE_RMS_0P2_SQRT_MAXDIM:
      return static_cast<float>(0.2 * std::sqrt(double(std::max(r, c))));
    default:
      return 1.f;
  }
}

size_t esize(int dt) { return dt == MUON_F32 ? 4 : 2; }

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Run the whole step (step_mode) or an NS-only pass over `reqs`.
// NS-only: reqs[i].G is the input, reqs[i].W the output (dtype w_dtype).
muon_status_t run(const std::vector<Req>& reqs, bool step_mode, float mu, int nesterov, float lr,
                  float wd, int scale_rule, const NsCfg& ns, cudaStream_t stream) {
  DevState* dev = nullptr;
  muon_status_t st = dev_state(&dev);
  if (st != MUON_OK) return st;
  const unsigned long long timeout_ns0 =
      static_cast<unsigned long long>(env_size("MUON_WAIT_TIMEOUT_MS", 2000)) * 1000000ull;
  Launcher L0{stream};

  // ---- small core shapes: one Gram-space kernel launch per core shape ---------------
  std::vector<Req> large;
  std::vector<SmallParams> smalls;
  {
    std::map<std::pair<int64_t, int64_t>, std::vector<int>> shapes;
    for (int i = 0; i < static_cast<int>(reqs.size()); ++i) {
      const Req& q = reqs[i];
      if (q.B <= 0 || q.m <= 0) continue;
      shapes[{q.m, q.n}].push_back(i);
    }
    for (auto& kv : shapes) {
      const int64_t m = kv.first.first, n = kv.first.second;
      if (!small_shape(m)) {
        const bool gs = gram_space_shape(m, n, ns);
        for (int i : kv.second) {
          large.push_back(reqs[i]);
          large.back().gs = gs;
        }
        continue;
      }
      for (size_t b = 0; b < kv.second.size(); b += kSmallMaxSlices) {
        smalls.emplace_back();
        SmallParams& sp = smalls.back();
        std::memset(&sp, 0, sizeof(sp));
        int64_t mats = 0;
        const size_t e = std::min(kv.second.size(), b + kSmallMaxSlices);
        for (size_t k = b; k < e; ++k) {
          const Req& q = reqs[kv.second[k]];
          SmallSlice& ss = sp.s[k - b];
          ss.G = q.G;
          ss.Mom = step_mode ? q.Mom : nullptr;
          ss.W = q.W;
          ss.count = static_cast<int>(q.B);
          ss.mat_base = static_cast<int>(mats);
          ss.trans = q.trans ? 1 : 0;
          ss.g_dtype = q.g_dtype;
          ss.w_dtype = q.w_dtype;
          ss.scale = scale_value(q.r, q.c, scale_rule);
          mats += q.B;
        }
        if (mats * cdiv(n, 128) >= (1LL << 31)) return MUON_ERR_UNSUPPORTED;
        sp.n_slices = static_cast<int>(e - b);
        int esg = 2, esw = 2;
        for (size_t k = b; k < e; ++k) {
          esg = std::max(esg, static_cast<int>(esize(reqs[kv.second[k]].g_dtype)));
          esw = std::max(esw, static_cast<int>(esize(reqs[kv.second[k]].w_dtype)));
        }
        if (!small_plan(m, n, mats, dev->sms, esg, esw, step_mode, ns.precise, &sp))
          return MUON_ERR_UNSUPPORTED;
        // TMA tile maps (stored layout): rows of 16-byte multiples, 16-byte
        // aligned bases; otherwise the kernel copies element-wise
        for (size_t k = b; k < e; ++k) {
          const Req& q = reqs[kv.second[k]];
          SmallSlice& ss = sp.s[k - b];
          const int bi_g = q.trans ? sp.m : sp.cw1, br_g = q.trans ? sp.cw1 : sp.m;
          const int bi_w = q.trans ? sp.m : 128, br_w = q.trans ? 128 : sp.m;
          auto legal = [&](const void* ptr, int dt, int box_inner) {
            const int64_t es = static_cast<int64_t>(esize(dt));
            return aligned(ptr, 16) && (q.c * es) % 16 == 0 && (box_inner * es) % 16 == 0;
          };
          ss.gbulk = legal(q.G, q.g_dtype, bi_g) && (!step_mode || legal(q.Mom, MUON_F32, bi_g)) &&
                     make_tile_map(&sp.tm[k - b][0], q.G, q.g_dtype, q.c, q.r, q.B, bi_g, br_g) &&
                     (!step_mode ||
                      make_tile_map(&sp.tm[k - b][1], q.Mom, MUON_F32, q.c, q.r, q.B, bi_g, br_g));
          ss.wbulk = legal(q.W, q.w_dtype, bi_w) &&
                     make_tile_map(&sp.tm[k - b][2], q.W, q.w_dtype, q.c, q.r, q.B, bi_w, br_w);
        }
        sp.steps = ns.steps;
        for (int it = 0; it < ns.steps; ++it) {
          sp.coef[it][0] = ns.coeffs[3 * it];
          sp.coef[it][1] = ns.coeffs[3 * it + 1];
          sp.coef[it][2] = ns.coeffs[3 * it + 2];
        }
        sp.step_mode = step_mode ? 1 : 0;
        sp.nesterov = nesterov ? 1 : 0;
        sp.mu = mu;
        sp.lr = lr;
        sp.wd = wd;
        sp.eps = ns.eps;
        sp.status = dev->status;
        sp.timeout_ns = timeout_ns0;
        sp.inject = take_injected_stall(kInjectSmall);
      }
    }
  }
  const size_t guard = env_size("MUON_WS_GUARD", 0) ? kGuardBytes : 0;
  std::vector<ChunkP> plan = make_plan(large, dev->sms, ns.precise, guard);
  size_t need = 0, need_ctr = 0, max_mats = 0;
  for (const SmallParams& sp : smalls) {
    size_t off[3], bands[3];
    need = std::max(need, small_ws_layout(sp, guard, off, bands));
    max_mats = std::max(max_mats, static_cast<size_t>(sp.total_mats));
  }
  for (auto& ch : plan) {
    need = std::max(need, ch.bytes);
    need_ctr = std::max(need_ctr, ch.ctrs);
  }
  if (smalls.empty() && plan.empty()) {
    t_last_launches = 0;
    return MUON_OK;
  }
  char* ws = nullptr;
  unsigned* ctr = nullptr;
  st = get_workspace(stream, need, need_ctr, &ws, &ctr);
  if (st != MUON_OK) return st;
  if (guard) {
    st = guard_counter(dev);
    if (st != MUON_OK) return st;
  }
  for (SmallParams& sp : smalls) {
    // the launches run in stream order, so each reuses the same workspace
    size_t off[3], bands[3];
    small_ws_layout(sp, guard, off, bands);
    sp.ximg = reinterpret_cast<uint8_t*>(ws + off[0]);
    sp.part = reinterpret_cast<float*>(ws + off[1]);
    sp.qimg = reinterpret_cast<uint8_t*>(ws + off[2]);
    if (guard) {
      st = guard_fill(ws, std::vector<size_t>(bands, bands + 3), guard, stream);
      if (st != MUON_OK) return st;
    }
    st = get_epoch_ctrs(stream, max_mats, &sp.arrive, &sp.ready_list, &sp.ctr, &sp.epoch, &sp.cap);
    if (st != MUON_OK) return st;
    // one CTA per SM (all resident: the launch is cooperative)
    if (small_blocks_per_sm(sp.smem_bytes, sp.precise != 0) <= 0) return MUON_ERR_CUDA;
    const int grid = static_cast<int>(std::min<int64_t>(sp.items, dev->sms));
    st = L0.run(5, [&] { return launch_small(sp, grid, stream); });
    if (st != MUON_OK) return st;
    if (guard) {
      st = guard_check(ws, std::vector<size_t>(bands, bands + 3), guard, dev, stream);
      if (st != MUON_OK) return st;
    }
  }
  if (plan.empty()) {
    t_last_launches = L0.count;
    return MUON_OK;
  }
  const unsigned long long timeout_ns =
      static_cast<unsigned long long>(env_size("MUON_WAIT_TIMEOUT_MS", 2000)) * 1000000ull;

  Launcher L{stream};
  for (const ChunkP& ch : plan) {
    if (guard) {
      st = guard_fill(ws, ch.guards, guard, stream);
      if (st != MUON_OK) return st;
    }
    // ---- K1 -------------------------------------------------------------------
    {
      PrepParams pp;
      std::memset(&pp, 0, sizeof(pp));
      int64_t blocks = 0;
      for (size_t i = 0; i < ch.slices.size(); ++i) {
        const SliceP& s = ch.slices[i];
        const Req& q = large[s.req];
        const NsGroupP& g = ch.groups[s.ng];
        PrepSlice& ps = pp.s[i];
        const int64_t per = q.r * q.c;
        ps.G = static_cast<const char*>(q.G) + s.b0 * per * esize(q.g_dtype);
        ps.Mom = step_mode ? q.Mom + s.b0 * per : nullptr;
        // the NS operand is kept as Xt = X^T: the stored layout when rows > cols
        auto* Xt = reinterpret_cast<__nv_bfloat16*>(ws + g.off_Xt0) + s.idx0 * g.n * g.m_pad;
        ps.direct = q.trans ? Xt : nullptr;
        ps.transp = q.trans ? nullptr : Xt;
        if (ns.precise) {
          auto* Xl = reinterpret_cast<__nv_bfloat16*>(ws + g.off_lo) + s.idx0 * g.n * g.m_pad;
          ps.direct_lo = q.trans ? Xl : nullptr;
          ps.transp_lo = q.trans ? nullptr : Xl;
        }
        ps.pitch_d = ps.pitch_t = g.m_pad;
        ps.mstride_d = ps.mstride_t = g.n * g.m_pad;
        ps.ssq_part = reinterpret_cast<float*>(ws + g.off_ssq) + s.idx0 * g.prep_tiles;
        ps.inv = reinterpret_cast<float*>(ws + g.off_inv) + s.idx0;
        ps.cnt = ctr + g.ctr_prep + s.idx0;
        ps.r = q.r;
        ps.c = q.c;
        ps.count = static_cast<int>(s.cnt);
        ps.g_dtype = q.g_dtype;
        ps.tiles_r = static_cast<int>(cdiv(q.r, kPrepTile));
        ps.tiles_c = static_cast<int>(cdiv(q.c, kPrepTile));
        ps.tile_base = static_cast<int>(blocks);
        const bool gvec = q.g_dtype == MUON_F32 ? (q.c % 4 == 0) : (q.c % 8 == 0);
        ps.vec = gvec && aligned(ps.G, 16) && (!step_mode || aligned(ps.Mom, 16));
        ps.trans = q.trans ? 1 : 0;
        blocks += s.cnt * ps.tiles_r * ps.tiles_c;
      }
      if (blocks >= (1LL << 31)) return MUON_ERR_UNSUPPORTED;
      pp.n_slices = static_cast<int>(ch.slices.size());
      pp.total_blocks = static_cast<int>(blocks);
      pp.step_mode = step_mode ? 1 : 0;
      pp.mu = mu;
      pp.nesterov = nesterov ? 1 : 0;
      pp.eps = ns.eps;
      pp.status = dev->status;
      st = L.run(0, [&] { return launch_prep(pp, stream); });
      if (st != MUON_OK) return st;
    }
    // ---- tensor maps -------------------------------------------------------------
    std::vector<NsGroupDev> dg(ch.groups.size());
    for (size_t k = 0; k < ch.groups.size(); ++k) {
      const NsGroupP& g = ch.groups[k];
      NsGroupDev& d = dg[k];
      d.m = g.m;
      d.n = g.n;
      d.cnt = g.cnt;
      d.m_pad = g.m_pad;
      d.Xt[0] = reinterpret_cast<__nv_bfloat16*>(ws + g.off_Xt0);
      d.Xt[1] = reinterpret_cast<__nv_bfloat16*>(ws + g.off_Xt1);
      d.A = reinterpret_cast<__nv_bfloat16*>(ws + g.off_A);
      d.B = reinterpret_cast<__nv_bfloat16*>(ws + g.off_B);
      d.inv = reinterpret_cast<const float*>(ws + g.off_inv);
      d.partial = reinterpret_cast<float*>(ws + g.off_part);
      d.tile_cnt = ctr + g.ctr_tile;
      d.ksplit = g.ksplit;
      d.kb_per_split = g.kb_per_split;
      d.num_kb_gram = g.num_kb_gram;
      d.tri = g.tri;
      if (ns.precise) {
        const size_t xb = align_up(static_cast<size_t>(g.cnt * g.n * g.m_pad) * 2, 1024);
        const size_t ab = align_up(static_cast<size_t>(g.cnt * g.m * g.m_pad) * 2, 1024);
        char* lo = ws + g.off_lo;
        d.Xt_lo[0] = reinterpret_cast<__nv_bfloat16*>(lo);
        d.Xt_lo[1] = reinterpret_cast<__nv_bfloat16*>(lo + xb);
        d.A_lo = reinterpret_cast<__nv_bfloat16*>(lo + 2 * xb);
        d.B_lo = reinterpret_cast<__nv_bfloat16*>(lo + 2 * xb + ab);
      }
      if (ch.gs) {
        d.gram_space = 1;
        for (int i = 0; i < 5; ++i) d.S[i] = reinterpret_cast<__nv_bfloat16*>(ws + g.off_S[i]);
        if (!ns_gs_maps(d)) return MUON_ERR_CUDA;
      }
      if (!ns_group_maps(d)) return MUON_ERR_CUDA;
    }
    // One grouped GEMM launch of product `epi` over every group of the chunk:
    // fill(G, group, first tile, mode) sets the groups' descriptors for single
    // tiles (mode 0), CTA pairs (1) or WIDE blocks (2); pairs or WIDE blocks
    // when the launch qualifies (bf16 products, no split-K; ns_plan.cpp).
    auto gemm = [&](int epi, auto&& fill, float a, float b, float c, float alpha,
                    int first) -> muon_status_t {
      GemmParams gp;
      std::memset(&gp, 0, sizeof(gp));
      int64_t tiles = 0;
      int min_kb = 1 << 30;
      bool split = false;
      int64_t min_m = INT64_MAX;
      double kb_sum = 0.0;
      for (size_t k = 0; k < ch.groups.size(); ++k) {
        GemmGroup& G = gp.g[k];
        fill(G, dg[k], static_cast<int>(tiles), 0);
        const int64_t gt = static_cast<int64_t>(G.tiles_per_mat) * dg[k].cnt;
        tiles += gt;
        kb_sum += static_cast<double>(gt) * G.kb_per_split;
        min_kb = std::min(min_kb, G.kb_per_split);
        split = split || G.ksplit > 1;
        min_m = std::min(min_m, dg[k].m);
      }
      const double mean_kb = tiles > 0 ? kb_sum / static_cast<double>(tiles) : 0.0;
      int mode = 0;
      if (!ns.precise && !split && gemm_use_wide(epi, tiles, dev->sms, min_kb, mean_kb))
        mode = 2;
      else if (!ns.precise && !split && gemm_use_pair(tiles, dev->sms, min_m))
        mode = 1;
      if (mode) {
        gp.pair = mode == 1 ? 1 : 0;
        gp.wide = mode == 2 ? 1 : 0;
        tiles = 0;
        for (size_t k = 0; k < ch.groups.size(); ++k) {
          fill(gp.g[k], dg[k], static_cast<int>(tiles), mode);
          tiles += static_cast<int64_t>(gp.g[k].tiles_per_mat) * dg[k].cnt;
        }
      }
      gp.deep = gemm_deep(epi, min_kb);
      gp.prec = ns.precise ? 1 : 0;
      if (const char* d = std::getenv("MUON_GEMM_DEEP")) gp.deep = d[0] == '1';   // tuning override
      if (tiles >= (1LL << 31)) return MUON_ERR_UNSUPPORTED;
      gp.n_groups = static_cast<int>(ch.groups.size());
      gp.total_tiles = static_cast<int>(tiles);
      gp.a = a;
      gp.b = b;
      gp.c = c;
      gp.alpha = alpha;
      gp.first = first;
      gp.status = dev->status;
      gp.timeout_ns = timeout_ns;
      gp.inject = take_injected_stall(kInjectGemm);
      gp.b_mn = ch.gs && epi != kEpiGram ? 1 : 0;   // Gram space: true products A B
      return L.run(1 + epi, [&] { return launch_gemm(epi, gp, stream); });
    };
    if (ch.gs) {
      // ---- NS in Gram space (ns_plan.cpp): per phase of `period` steps the Gram
      // R of the iterate, then per step B'_k, Q, T, R_{k+1}; the phase ends with
      // the apply X <- Q X (the first one also scales by 1 / ||X0||).
      auto sym = [](int a, int b, int c) {
        return [a, b, c](GemmGroup& G, const NsGroupDev& d, int base, int mode) {
          ns_fill_gs_sym(G, d, a, b, c, base, mode == 1, mode == 2);
        };
      };
      int64_t gs_min_m = INT64_MAX;   // one period per chunk: its smallest m decides
      for (const NsGroupP& g : ch.groups) gs_min_m = std::min(gs_min_m, g.m);
      const int period = gram_restart_period(gs_min_m);
      int src = 0;   // Xt buffer holding the iterate
      for (int k0 = 0; k0 < ns.steps; k0 += period) {
        const int k1 = std::min(ns.steps, k0 + period);
        st = gemm(kEpiGram, [src](GemmGroup& G, const NsGroupDev& d, int base, int mode) {
                    ns_fill_gs_gram(G, d, src, base, mode == 1, mode == 2);
                  }, 0.f, 0.f, 0.f, 0.f, k0 == 0 ? 1 : 0);
        if (st != MUON_OK) return st;
        int q = kGsQ0;
        for (int it = k0; it < k1; ++it) {
          const float ca = ns.coeffs[3 * it], cb = ns.coeffs[3 * it + 1], cc = ns.coeffs[3 * it + 2];
          const float alpha = kShiftFrac * ca;
          const bool more = it + 1 < k1;
          if (it > k0 || more) {   // B'_k = b R + c R^2 + alpha I
            st = gemm(kEpiPoly, sym(kGsR, kGsR, kGsB), 0.f, cb, cc, alpha, 0);
            if (st != MUON_OK) return st;
          }
          if (it == k0) {          // Q = P_k = a I + b R_k + c R_k^2
            st = gemm(kEpiPoly, sym(kGsR, kGsR, q), 0.f, cb, cc, ca, 0);
          } else {                 // Q <- (a - alpha) Q + Q B'_k
            st = gemm(kEpiPoly, sym(q, kGsB, 2 * kGsQ0 + 1 - q), 0.f, ca - alpha, 1.f, 0.f, 0);
            q = 2 * kGsQ0 + 1 - q;
          }
          if (st != MUON_OK) return st;
          if (more) {              // T = (a - alpha) R + R B'; R_{k+1} = (a - alpha) T + T B'
            st = gemm(kEpiPoly, sym(kGsR, kGsB, kGsT), 0.f, ca - alpha, 1.f, 0.f, 0);
            if (st != MUON_OK) return st;
            st = gemm(kEpiPoly, sym(kGsT, kGsB, kGsR), 0.f, ca - alpha, 1.f, 0.f, 0);
            if (st != MUON_OK) return st;
          }
        }
        // X <- Q X (the first phase: Q X0 / ||X0||) into the other Xt buffer
        st = gemm(kEpiApply, [q, src](GemmGroup& G, const NsGroupDev& d, int base, int mode) {
                    ns_fill_gs_apply(G, d, q, src, base, mode == 1, mode == 2);
                  }, 0.f, 0.f, 0.f, 0.f, k0 == 0 ? 1 : 0);
        if (st != MUON_OK) return st;
        src ^= 1;
      }
    }
    // ---- NS iterations (X space) -------------------------------------------------
    for (int it = 0; !ch.gs && it < ns.steps; ++it) {
      const float ca = ns.coeffs[3 * it], cb = ns.coeffs[3 * it + 1], cc = ns.coeffs[3 * it + 2];
      // X' = a X + (b A + c A^2) X is evaluated as (a - alpha) X + (B + alpha I) X:
      // identical in exact arithmetic, but the bf16 operand B + alpha I is
      // smaller where a X and B X cancel, which lowers the rounding error.
      const float alpha = kShiftFrac * ca;
      for (int phase = 0; phase < 3; ++phase) {
        st = gemm(phase, [phase, it](GemmGroup& G, const NsGroupDev& d, int base, int mode) {
                    ns_fill_group(G, d, phase, it, base, mode == 1, mode == 2);
                  }, ca - alpha, cb, cc, alpha, it == 0 ? 1 : 0);
        if (st != MUON_OK) return st;
      }
    }
    // ---- K6 -------------------------------------------------------------------
    {
      int64_t chunk_min_m = INT64_MAX;   // the Gram-space restart period's m
      for (const NsGroupP& g : ch.groups) chunk_min_m = std::min(chunk_min_m, g.m);
      FinParams fp;
      std::memset(&fp, 0, sizeof(fp));
      fp.passes = fin_passes(ch.slices, large);
      int64_t blocks = 0;
      for (size_t i = 0; i < ch.slices.size(); ++i) {
        const SliceP& s = ch.slices[i];
        const Req& q = large[s.req];
        const NsGroupP& g = ch.groups[s.ng];
        FinSlice& fs = fp.s[i];
        const int64_t per = q.r * q.c;
        fs.W = static_cast<char*>(q.W) + s.b0 * per * esize(q.w_dtype);
        // the Xt buffer of the result: one per step (X space) or per phase (Gram space)
        const int fin = (ch.gs ? gram_phases(ns.steps, chunk_min_m) : ns.steps) & 1;
        // O = Xt in the stored layout when rows > cols, else its transpose
        fs.O = reinterpret_cast<__nv_bfloat16*>(ws + (fin ? g.off_Xt1 : g.off_Xt0)) +
               s.idx0 * g.n * g.m_pad;
        if (ns.precise)
          fs.O_lo = reinterpret_cast<__nv_bfloat16*>(
                        ws + g.off_lo +
                        (fin ? align_up(static_cast<size_t>(g.cnt * g.n * g.m_pad) * 2, 1024) : 0)) +
                    s.idx0 * g.n * g.m_pad;
        fs.o_trans = q.trans ? 0 : 1;
        fs.pitch_o = g.m_pad;
        fs.mstride_o = g.n * g.m_pad;
        fs.inv = ns.steps == 0 ? reinterpret_cast<const float*>(ws + g.off_inv) + s.idx0
                               : nullptr;
        fs.r = q.r;
        fs.c = q.c;
        fs.count = static_cast<int>(s.cnt);
        fs.w_dtype = q.w_dtype;
        fs.tiles_r = static_cast<int>(cdiv(q.r, fin_tile_rows(fs.o_trans, fp.passes)));
        fs.tiles_c = static_cast<int>(cdiv(q.c, fs.o_trans ? kFinTCols : kFinCols));
        fs.tile_base = static_cast<int>(blocks);
        fs.vec = (q.w_dtype == MUON_F32 ? (q.c % 4 == 0) : (q.c % 8 == 0)) && aligned(fs.W, 16);
        fs.scale = scale_value(q.r, q.c, scale_rule);
        blocks += s.cnt * fs.tiles_r * fs.tiles_c;
      }
      if (blocks >= (1LL << 31)) return MUON_ERR_UNSUPPORTED;
      fp.n_slices = static_cast<int>(ch.slices.size());
      fp.total_blocks = static_cast<int>(blocks);
      fp.status = dev->status;
      fp.step_mode = step_mode ? 1 : 0;
      fp.lr = lr;
      fp.wd = wd;
      st = L.run(4, [&] { return launch_finish(fp, stream); });
      if (st != MUON_OK) return st;
    }
    if (guard) {
      st = guard_check(ws, ch.guards, guard, dev, stream);
      if (st != MUON_OK) return st;
    }
  }
  t_last_launches = L.count + L0.count;
  return MUON_OK;
}

bool ranges_overlap(const std::vector<std::pair<uintptr_t, uintptr_t>>& r) {
  std::vector<std::pair<uintptr_t, uintptr_t>> v;
  for (auto& x : r)
    if (x.second > x.first) v.push_back(x);
  std::sort(v.begin(), v.end());
  for (size_t i = 1; i < v.size(); ++i)
    if (v[i].first < v[i - 1].second) return true;
  return false;
}

muon_status_t step_impl(const muon_group_t* groups, int n_groups, float mu, int nesterov,
                        float lr, float wd, int scale_rule, const muon_ns_config_t* nscfg,
                        cudaStream_t stream) {
  if (n_groups < 0 || (n_groups > 0 && !groups)) return MUON_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(mu) || !std::isfinite(lr) || !std::isfinite(wd))
    return MUON_ERR_INVALID_ARGUMENT;
  if (scale_rule < 0 || scale_rule > MUON_SCALE_ONE) return MUON_ERR_INVALID_ARGUMENT;
  NsCfg ns;
  muon_status_t st = check_ns_cfg(nscfg, &ns);
  if (st != MUON_OK) return st;
  std::vector<Req> reqs;
  std::vector<std::pair<uintptr_t, uintptr_t>> written, all;
  for (int i = 0; i < n_groups; ++i) {
    const muon_group_t& g = groups[i];
    if (g.B < 0 || g.M < 0 || g.N < 0) return MUON_ERR_INVALID_ARGUMENT;
    if (g.w_dtype != MUON_F32 && g.w_dtype != MUON_BF16) return MUON_ERR_INVALID_ARGUMENT;
    if (g.g_dtype != MUON_F32 && g.g_dtype != MUON_BF16) return MUON_ERR_INVALID_ARGUMENT;
    if (g.B == 0 || g.M == 0 || g.N == 0) continue;
    if (!g.W || !g.G || !g.Mom) return MUON_ERR_INVALID_ARGUMENT;
    if (!aligned(g.W, esize(g.w_dtype)) || !aligned(g.G, esize(g.g_dtype)) || !aligned(g.Mom, 4))
      return MUON_ERR_INVALID_ARGUMENT;
    if (g.M > (1LL << 30) || g.N > (1LL << 30) || g.B > (1LL << 30))
      return MUON_ERR_UNSUPPORTED;
    const int64_t per = g.M * g.N;
    const auto w0 = reinterpret_cast<uintptr_t>(g.W);
    const auto g0 = reinterpret_cast<uintptr_t>(g.G);
    const auto m0 = reinterpret_cast<uintptr_t>(g.Mom);
    const uintptr_t wl = static_cast<uintptr_t>(g.B * per) * esize(g.w_dtype);
    const uintptr_t gl = static_cast<uintptr_t>(g.B * per) * esize(g.g_dtype);
    const uintptr_t ml = static_cast<uintptr_t>(g.B * per) * 4;
    written.push_back({w0, w0 + wl});
    written.push_back({m0, m0 + ml});
    // a G range may be shared by two groups, but never with a written range
    for (auto& x : std::vector<std::pair<uintptr_t, uintptr_t>>{{w0, w0 + wl}, {m0, m0 + ml}})
      if (g0 < x.second && x.first < g0 + gl) return MUON_ERR_ALIAS;
    all.push_back({g0, g0 + gl});
    Req q;
    q.W = g.W;
    q.w_dtype = g.w_dtype;
    q.G = g.G;
    q.g_dtype = g.g_dtype;
    q.Mom = g.Mom;
    q.B = g.B;
    q.r = g.M;
    q.c = g.N;
    q.trans = g.M > g.N;
    q.m = std::min(g.M, g.N);
    q.n = std::max(g.M, g.N);
    reqs.push_back(q);
  }
  if (ranges_overlap(written)) return MUON_ERR_ALIAS;
  for (auto& gr : all)
    for (auto& w : written)
      if (gr.first < w.second && w.first < gr.second) return MUON_ERR_ALIAS;
  if (reqs.empty()) {
    t_last_launches = 0;
    return MUON_OK;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  return run(reqs, true, mu, nesterov, lr, wd, scale_rule, ns, stream);
}

muon_status_t ns_impl(void* X, int dtype, int64_t B, int64_t M, int64_t N,
                      const muon_ns_config_t* cfg, void* out, cudaStream_t stream) {
  if (B < 0 || M < 0 || N < 0) return MUON_ERR_INVALID_ARGUMENT;
  if (dtype != MUON_F32 && dtype != MUON_BF16) return MUON_ERR_INVALID_ARGUMENT;
  NsCfg ns;
  muon_status_t st = check_ns_cfg(cfg, &ns);
  if (st != MUON_OK) return st;
  if (B == 0 || M == 0 || N == 0) {
    t_last_launches = 0;
    return MUON_OK;
  }
  if (!X) return MUON_ERR_INVALID_ARGUMENT;
  if (!aligned(X, esize(dtype)) || (out && !aligned(out, esize(dtype))))
    return MUON_ERR_INVALID_ARGUMENT;
  if (M > (1LL << 30) || N > (1LL << 30) || B > (1LL << 30)) return MUON_ERR_UNSUPPORTED;
  const uintptr_t len = static_cast<uintptr_t>(B * M * N) * esize(dtype);
  if (out && out != X) {
    const auto x0 = reinterpret_cast<uintptr_t>(X), o0 = reinterpret_cast<uintptr_t>(out);
    if (x0 < o0 + len && o0 < x0 + len) return MUON_ERR_ALIAS;
  }
  Req q;
  q.W = out ? out : X;
  q.w_dtype = dtype;
  q.G = X;
  q.g_dtype = dtype;
  q.Mom = nullptr;
  q.B = B;
  q.r = M;
  q.c = N;
  q.trans = M > N;
  q.m = std::min(M, N);
  q.n = std::max(M, N);
  std::lock_guard<std::mutex> lock(g_mu);
  return run({q}, false, 0.f, 0, 0.f, 0.f, MUON_SCALE_ONE, ns, stream);
}

// ---- host-resident state ------------------------------------------------------------
// One Muon step over parameters whose W, G and Mom live in host memory.  The
// matrices are cut into up to 8 chunks of at least 20 MB (the first and last
// half the size of the others: weights 1, 2, ..., 2, 1); chunk i moves
// through device slot i % 3: copy-in on one stream, the step on a second,
// copy-out (W', Mom') on a third, so that the two copy directions and the
// kernels overlap.  Everything is ordered after the work already on
// `stream`, and `stream` waits for the last copy-out: the call is
// asynchronous on `stream` like the device entry points.
muon_status_t host_pipe(cudaStream_t stream, size_t slot_bytes, HostPipe** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_CUDA;
  HostPipe& h = g_host[{dev, stream}];
  if (!h.s_in) {
    for (cudaStream_t* st : {&h.s_in, &h.s_comp, &h.s_out})
      if (cudaStreamCreateWithFlags(st, cudaStreamNonBlocking) != cudaSuccess) return MUON_ERR_CUDA;
    if (cudaEventCreateWithFlags(&h.ev_start, cudaEventDisableTiming) != cudaSuccess)
      return MUON_ERR_CUDA;
    for (int i = 0; i < kHostSlots; ++i)
      for (cudaEvent_t* e : {&h.ev_in[i], &h.ev_comp[i], &h.ev_free[i]})
        if (cudaEventCreateWithFlags(e, cudaEventDisableTiming) != cudaSuccess) return MUON_ERR_CUDA;
  }
  if (h.slot_bytes < slot_bytes) {
    // earlier calls may still use the old slots
    for (cudaStream_t st : {h.s_in, h.s_comp, h.s_out})
      if (cudaStreamSynchronize(st) != cudaSuccess) return MUON_ERR_CUDA;
    if (h.slot) cudaFree(h.slot);
    h.slot = nullptr;
    h.slot_bytes = 0;
    const size_t want = align_up(slot_bytes, size_t(1) << 21);
    if (cudaMalloc(&h.slot, want * kHostSlots) != cudaSuccess) {
      cudaGetLastError();
      h.slot = nullptr;
      return MUON_ERR_OUT_OF_MEMORY;
    }
    h.slot_bytes = want;
  }
  *out = &h;
  return MUON_OK;
}

muon_status_t host_step_impl(const muon_group_t* groups, int n_groups, float mu, int nesterov,
                             float lr, float wd, int scale_rule, const muon_ns_config_t* nscfg,
                             cudaStream_t stream) {
  if (n_groups < 0 || (n_groups > 0 && !groups)) return MUON_ERR_INVALID_ARGUMENT;
  if (!std::isfinite(mu) || !std::isfinite(lr) || !std::isfinite(wd))
    return MUON_ERR_INVALID_ARGUMENT;
  if (scale_rule < 0 || scale_rule > MUON_SCALE_ONE) return MUON_ERR_INVALID_ARGUMENT;
  NsCfg ns;
  muon_status_t st = check_ns_cfg(nscfg, &ns);
  if (st != MUON_OK) return st;
  // validation and alias rules of the device entry point, on host ranges
  std::vector<std::pair<uintptr_t, uintptr_t>> written, all;
  struct Unit {
    int g;
    size_t bytes;   // W + G + Mom of one matrix
  };
  std::vector<Unit> units;
  size_t total = 0;
  for (int i = 0; i < n_groups; ++i) {
    const muon_group_t& g = groups[i];
    if (g.B < 0 || g.M < 0 || g.N < 0) return MUON_ERR_INVALID_ARGUMENT;
    if (g.w_dtype != MUON_F32 && g.w_dtype != MUON_BF16) return MUON_ERR_INVALID_ARGUMENT;
    if (g.g_dtype != MUON_F32 && g.g_dtype != MUON_BF16) return MUON_ERR_INVALID_ARGUMENT;
    if (g.B == 0 || g.M == 0 || g.N == 0) continue;
    if (!g.W || !g.G || !g.Mom) return MUON_ERR_INVALID_ARGUMENT;
    if (!aligned(g.W, esize(g.w_dtype)) || !aligned(g.G, esize(g.g_dtype)) || !aligned(g.Mom, 4))
      return MUON_ERR_INVALID_ARGUMENT;
    if (g.M > (1LL << 30) || g.N > (1LL << 30) || g.B > (1LL << 30))
      return MUON_ERR_UNSUPPORTED;
    const size_t per = static_cast<size_t>(g.M * g.N);
    const auto w0 = reinterpret_cast<uintptr_t>(g.W);
    const auto g0 = reinterpret_cast<uintptr_t>(g.G);
    const auto m0 = reinterpret_cast<uintptr_t>(g.Mom);
    const uintptr_t wl = g.B * per * esize(g.w_dtype), gl = g.B * per * esize(g.g_dtype),
                    ml = g.B * per * 4;
    written.push_back({w0, w0 + wl});
    written.push_back({m0, m0 + ml});
    for (auto& x : std::vector<std::pair<uintptr_t, uintptr_t>>{{w0, w0 + wl}, {m0, m0 + ml}})
      if (g0 < x.second && x.first < g0 + gl) return MUON_ERR_ALIAS;
    all.push_back({g0, g0 + gl});
    const size_t ub = per * (esize(g.w_dtype) + esize(g.g_dtype) + 4);
    for (int64_t b = 0; b < g.B; ++b) units.push_back({i, ub});
    total += g.B * ub;
  }
  if (ranges_overlap(written)) return MUON_ERR_ALIAS;
  for (auto& gr : all)
    for (auto& w : written)
      if (gr.first < w.second && w.first < gr.second) return MUON_ERR_ALIAS;
  if (units.empty()) {
    t_last_launches = 0;
    return MUON_OK;
  }
  // chunks: consecutive matrices (at least one per chunk); a segment is a run
  // of one group's matrices
  struct Seg {
    int g;
    int64_t b0, cnt;
  };
  std::vector<std::vector<Seg>> chunks;
  // K chunks, K = total / 20 MB clamped to [1, 8] (MUON_HOST_CHUNKS overrides
  // the 8): each chunk costs its launches (tens of microseconds on the small-m
  // path).  The pipeline fills with the first chunk's copy-in and drains with
  // the last one's copy-out, so those two are half the size of the others
  // (weights 1, 2, ..., 2, 1).  A chunk closes once the bytes so far reach
  // its cumulative boundary; every chunk holds at least one matrix.  On
  // 74 x [24, 10240] (327 MB of state) 7 / 8 / 15 chunks took 1.32 / 1.28 /
  // 1.28 ms, and four or six device slots instead of three under 1 % less.
  const size_t kmax = std::max<size_t>(env_size("MUON_HOST_CHUNKS", 8), 1);
  const size_t K = std::min(kmax, std::max<size_t>(total / (size_t(20) << 20), 1));
  std::vector<double> bound(K);
  {
    const double wsum = K == 1 ? 1.0 : static_cast<double>(2 * (K - 1));
    double acc = 0.0;
    for (size_t i = 0; i < K; ++i) {
      acc += (K == 1) ? 1.0 : ((i == 0 || i == K - 1) ? 1.0 : 2.0);
      bound[i] = acc / wsum * static_cast<double>(total);
    }
  }
  {
    std::vector<Seg> cur;
    size_t done = 0;
    int64_t next_b = 0;
    int prev_g = -1;
    for (const Unit& u : units) {
      if (u.g != prev_g) next_b = 0;
      if (!cur.empty() && chunks.size() + 1 < K &&
          static_cast<double>(done) >= bound[chunks.size()] - 0.5 * u.bytes) {
        chunks.push_back(cur);
        cur.clear();
      }
      if (!cur.empty() && cur.back().g == u.g && cur.back().b0 + cur.back().cnt == next_b)
        ++cur.back().cnt;
      else
        cur.push_back({u.g, next_b, 1});
      done += u.bytes;
      ++next_b;
      prev_g = u.g;
    }
    if (!cur.empty()) chunks.push_back(cur);
  }
  // slot layout of a chunk: per segment W, G, Mom, each 256-byte aligned
  auto seg_bytes = [&](const Seg& sg, size_t* ow, size_t* og, size_t* om, size_t off) {
    const muon_group_t& g = groups[sg.g];
    const size_t e = static_cast<size_t>(sg.cnt * g.M * g.N);
    *ow = off;
    *og = align_up(*ow + e * esize(g.w_dtype), 256);
    *om = align_up(*og + e * esize(g.g_dtype), 256);
    return align_up(*om + e * 4, 256);
  };
  size_t slot_need = 256;
  for (auto& ch : chunks) {
    size_t off = 0, a, b, c;
    for (auto& sg : ch) off = seg_bytes(sg, &a, &b, &c, off);
    slot_need = std::max(slot_need, off);
  }
  std::lock_guard<std::mutex> lock(g_mu);
  HostPipe* hp = nullptr;
  st = host_pipe(stream, slot_need, &hp);
  if (st != MUON_OK) return st;
  if (cudaEventRecord(hp->ev_start, stream) != cudaSuccess) return MUON_ERR_CUDA;
  for (cudaStream_t x : {hp->s_in, hp->s_comp, hp->s_out})
    if (cudaStreamWaitEvent(x, hp->ev_start, 0) != cudaSuccess) return MUON_ERR_CUDA;
  int launches = 0;
  for (size_t ci = 0; ci < chunks.size(); ++ci) {
    const int k = static_cast<int>(ci % kHostSlots);
    char* base = static_cast<char*>(hp->slot) + k * hp->slot_bytes;
    if (ci >= static_cast<size_t>(kHostSlots) &&
        cudaStreamWaitEvent(hp->s_in, hp->ev_free[k], 0) != cudaSuccess)
      return MUON_ERR_CUDA;
    std::vector<Req> reqs;
    size_t off = 0;
    for (const Seg& sg : chunks[ci]) {
      const muon_group_t& g = groups[sg.g];
      size_t ow, og, om;
      off = seg_bytes(sg, &ow, &og, &om, off);
      const size_t per = static_cast<size_t>(g.M * g.N);
      const size_t e = sg.cnt * per;
      const size_t h0 = static_cast<size_t>(sg.b0) * per;
      if (cudaMemcpyAsync(base + ow, static_cast<const char*>(g.W) + h0 * esize(g.w_dtype),
                          e * esize(g.w_dtype), cudaMemcpyHostToDevice, hp->s_in) != cudaSuccess ||
          cudaMemcpyAsync(base + og, static_cast<const char*>(g.G) + h0 * esize(g.g_dtype),
                          e * esize(g.g_dtype), cudaMemcpyHostToDevice, hp->s_in) != cudaSuccess ||
          cudaMemcpyAsync(base + om, g.Mom + h0, e * 4, cudaMemcpyHostToDevice, hp->s_in) !=
              cudaSuccess)
        return MUON_ERR_CUDA;
      Req q;
      q.W = base + ow;
      q.w_dtype = g.w_dtype;
      q.G = base + og;
      q.g_dtype = g.g_dtype;
      q.Mom = reinterpret_cast<float*>(base + om);
      q.B = sg.cnt;
      q.r = g.M;
      q.c = g.N;
      q.trans = g.M > g.N;
      q.m = std::min(g.M, g.N);
      q.n = std::max(g.M, g.N);
      reqs.push_back(q);
    }
    if (cudaEventRecord(hp->ev_in[k], hp->s_in) != cudaSuccess ||
        cudaStreamWaitEvent(hp->s_comp, hp->ev_in[k], 0) != cudaSuccess)
      return MUON_ERR_CUDA;
    st = run(reqs, true, mu, nesterov, lr, wd, scale_rule, ns, hp->s_comp);
    if (st != MUON_OK) return st;
    launches += t_last_launches;
    if (cudaEventRecord(hp->ev_comp[k], hp->s_comp) != cudaSuccess ||
        cudaStreamWaitEvent(hp->s_out, hp->ev_comp[k], 0) != cudaSuccess)
      return MUON_ERR_CUDA;
    off = 0;
    for (const Seg& sg : chunks[ci]) {
      const muon_group_t& g = groups[sg.g];
      size_t ow, og, om;
      off = seg_bytes(sg, &ow, &og, &om, off);
      const size_t per = static_cast<size_t>(g.M * g.N);
      const size_t e = sg.cnt * per;
      const size_t h0 = static_cast<size_t>(sg.b0) * per;
      if (cudaMemcpyAsync(static_cast<char*>(g.W) + h0 * esize(g.w_dtype), base + ow,
                          e * esize(g.w_dtype), cudaMemcpyDeviceToHost, hp->s_out) != cudaSuccess ||
          cudaMemcpyAsync(g.Mom + h0, base + om, e * 4, cudaMemcpyDeviceToHost, hp->s_out) !=
              cudaSuccess)
        return MUON_ERR_CUDA;
    }
    if (cudaEventRecord(hp->ev_free[k], hp->s_out) != cudaSuccess) return MUON_ERR_CUDA;
  }
  // the copy-out stream ran last for every chunk; the caller's stream waits for it
  const int last = static_cast<int>((chunks.size() - 1) % kHostSlots);
  if (cudaStreamWaitEvent(stream, hp->ev_free[last], 0) != cudaSuccess) return MUON_ERR_CUDA;
  t_last_launches = launches;
  return MUON_OK;
}

// ---- AdamW for the non-matrix parameters ----------------------------------------------
muon_status_t adamw_impl(const muon_adamw_group_t* groups, int n_groups,
                         const muon_adamw_config_t* cfg, cudaStream_t stream) {
  if (n_groups < 0 || (n_groups > 0 && !groups) || !cfg) return MUON_ERR_INVALID_ARGUMENT;
  const float hp[5] = {cfg->lr, cfg->beta1, cfg->beta2, cfg->eps, cfg->weight_decay};
  for (float x : hp)
    if (!std::isfinite(x)) return MUON_ERR_INVALID_ARGUMENT;
  if (cfg->beta1 < 0.f || cfg->beta1 >= 1.f || cfg->beta2 < 0.f || cfg->beta2 >= 1.f ||
      cfg->eps < 0.f || cfg->step < 1)
    return MUON_ERR_INVALID_ARGUMENT;
  std::vector<std::pair<uintptr_t, uintptr_t>> written, read;
  std::vector<int> live;
  for (int i = 0; i < n_groups; ++i) {
    const muon_adamw_group_t& g = groups[i];
    if (g.numel < 0) return MUON_ERR_INVALID_ARGUMENT;
    if (g.p_dtype != MUON_F32 && g.p_dtype != MUON_BF16) return MUON_ERR_INVALID_ARGUMENT;
    if (g.g_dtype != MUON_F32 && g.g_dtype != MUON_BF16) return MUON_ERR_INVALID_ARGUMENT;
    if (g.numel == 0) continue;
    if (!g.param || !g.grad || !g.exp_avg || !g.exp_avg_sq) return MUON_ERR_INVALID_ARGUMENT;
    if (!aligned(g.param, esize(g.p_dtype)) || !aligned(g.grad, esize(g.g_dtype)) ||
        !aligned(g.exp_avg, 4) || !aligned(g.exp_avg_sq, 4))
      return MUON_ERR_INVALID_ARGUMENT;
    if (g.numel > (int64_t(1) << 40)) return MUON_ERR_UNSUPPORTED;
    const auto pp = reinterpret_cast<uintptr_t>(g.param);
    const auto mp = reinterpret_cast<uintptr_t>(g.exp_avg);
    const auto vp = reinterpret_cast<uintptr_t>(g.exp_avg_sq);
    const auto gp = reinterpret_cast<uintptr_t>(g.grad);
    written.push_back({pp, pp + g.numel * esize(g.p_dtype)});
    written.push_back({mp, mp + g.numel * 4});
    written.push_back({vp, vp + g.numel * 4});
    read.push_back({gp, gp + g.numel * esize(g.g_dtype)});
    live.push_back(i);
  }
  if (ranges_overlap(written)) return MUON_ERR_ALIAS;
  for (auto& r : read)
    for (auto& w : written)
      if (r.first < w.second && w.first < r.second) return MUON_ERR_ALIAS;
  if (live.empty()) {
    t_last_launches = 0;
    return MUON_OK;
  }
  std::lock_guard<std::mutex> lock(g_mu);
  DevState* dev = nullptr;
  muon_status_t st = dev_state(&dev);
  if (st != MUON_OK) return st;
  // bias corrections in double: 1 - beta^t for large t is close to 1
  const double bc1 = 1.0 - std::pow(static_cast<double>(cfg->beta1), static_cast<double>(cfg->step));
  const double bc2 = 1.0 - std::pow(static_cast<double>(cfg->beta2), static_cast<double>(cfg->step));
  Launcher L{stream};
  for (size_t b = 0; b < live.size(); b += kMaxSlices) {
    AdamwParams ap;
    std::memset(&ap, 0, sizeof(ap));
    int64_t units = 0;
    const size_t e = std::min(live.size(), b + kMaxSlices);
    for (size_t k = b; k < e; ++k) {
      const muon_adamw_group_t& g = groups[live[k]];
      AdamwSlice& sl = ap.s[k - b];
      sl.p = g.param;
      sl.g = g.grad;
      sl.m = g.exp_avg;
      sl.v = g.exp_avg_sq;
      sl.numel = g.numel;
      sl.unit_base = units;
      sl.p_dtype = g.p_dtype;
      sl.g_dtype = g.g_dtype;
      sl.vec = aligned(g.param, 16) && aligned(g.grad, 16) && aligned(g.exp_avg, 16) &&
               aligned(g.exp_avg_sq, 16);
      units += cdiv(g.numel, 8);
    }
    ap.n_slices = static_cast<int>(e - b);
    ap.total_units = units;
    ap.lr = cfg->lr;
    ap.beta1 = cfg->beta1;
    ap.beta2 = cfg->beta2;
    ap.eps = cfg->eps;
    ap.wd = cfg->weight_decay;
    ap.step_size = static_cast<float>(static_cast<double>(cfg->lr) / bc1);
    ap.inv_sqrt_bc2 = static_cast<float>(1.0 / std::sqrt(bc2));
    st = L.run(6, [&] { return launch_adamw(ap, dev->sms, stream); });
    if (st != MUON_OK) return st;
  }
  t_last_launches = L.count;
  return MUON_OK;
}

}  // namespace

namespace muon {
int take_injected_stall(int kind) {
  int want = kind;
  return g_inject.compare_exchange_strong(want, 0) ? 1 : 0;
}
}  // namespace muon

extern "C" {

muon_status_t muon_ns_default_config(muon_ns_config_t* cfg) {
  if (!cfg) return MUON_ERR_INVALID_ARGUMENT;
  cfg->steps = kDefSteps;
  cfg->coeffs = nullptr;
  cfg->a = kDefA;
  cfg->b = kDefB;
  cfg->c = kDefC;
  cfg->eps = kDefEps;
  cfg->precision = MUON_NS_BF16;
  return MUON_OK;
}

muon_status_t muon_ns_batched(void* X, int64_t B, int64_t M, int64_t N, int steps, float a,
                              float b, float c, cudaStream_t stream) {
  muon_ns_config_t cfg;
  muon_ns_default_config(&cfg);
  cfg.steps = steps;
  cfg.a = a;
  cfg.b = b;
  cfg.c = c;
  try {
    return ns_impl(X, MUON_BF16, B, M, N, &cfg, nullptr, stream);
  } catch (...) {
    return MUON_ERR_OUT_OF_MEMORY;
  }
}

muon_status_t muon_ns_batched_ex(void* X, int32_t dtype, int64_t B, int64_t M, int64_t N,
                                 const muon_ns_config_t* cfg, void* out, cudaStream_t stream) {
  try {
    return ns_impl(X, dtype, B, M, N, cfg, out, stream);
  } catch (...) {
    return MUON_ERR_OUT_OF_MEMORY;
  }
}

muon_status_t muon_step_grouped(const muon_group_t* groups, int n_groups, float mu, int nesterov,
                                float lr, float wd, int scale_rule, cudaStream_t stream) {
  try {
    return step_impl(groups, n_groups, mu, nesterov, lr, wd, scale_rule, nullptr, stream);
  } catch (...) {
    return MUON_ERR_OUT_OF_MEMORY;
  }
}

muon_status_t muon_step_grouped_ex(const muon_group_t* groups, int n_groups, float mu,
                                   int nesterov, float lr, float wd, int scale_rule,
                                   const muon_ns_config_t* ns, cudaStream_t stream) {
  try {
    return step_impl(groups, n_groups, mu, nesterov, lr, wd, scale_rule, ns, stream);
  } catch (...) {
    return MUON_ERR_OUT_OF_MEMORY;
  }
}

muon_status_t muon_step_grouped_host(const muon_group_t* groups, int n_groups, float mu,
                                     int nesterov, float lr, float wd, int scale_rule,
                                     const muon_ns_config_t* ns, cudaStream_t stream) {
  try {
    return host_step_impl(groups, n_groups, mu, nesterov, lr, wd, scale_rule, ns, stream);
  } catch (...) {
    return MUON_ERR_OUT_OF_MEMORY;
  }
}

muon_status_t muon_adamw_grouped(const muon_adamw_group_t* groups, int n_groups,
                                 const muon_adamw_config_t* cfg, cudaStream_t stream) {
  try {
    return adamw_impl(groups, n_groups, cfg, stream);
  } catch (...) {
    return MUON_ERR_OUT_OF_MEMORY;
  }
}

muon_status_t muon_ns_cost_table(const int64_t* shapes, int n, const muon_ns_config_t* cfg,
                                 int reps, double* ms_per_matrix, cudaStream_t stream) {
  try {
    if (n < 0 || reps < 1 || (n > 0 && (!shapes || !ms_per_matrix)))
      return MUON_ERR_INVALID_ARGUMENT;
    for (int i = 0; i < n; ++i)
      if (shapes[2 * i] <= 0 || shapes[2 * i + 1] <= 0 || shapes[2 * i] > (1LL << 30) ||
          shapes[2 * i + 1] > (1LL << 30))
        return MUON_ERR_INVALID_ARGUMENT;
    if (n == 0) return MUON_OK;
    void* buf = nullptr;
    size_t have = 0;
    cudaEvent_t e0 = nullptr, e1 = nullptr;
    if (cudaEventCreate(&e0) != cudaSuccess || cudaEventCreate(&e1) != cudaSuccess)
      return MUON_ERR_CUDA;
    muon_status_t st = MUON_OK;
    for (int i = 0; i < n && st == MUON_OK; ++i) {
      const int64_t r = shapes[2 * i], c = shapes[2 * i + 1];
      const size_t per = static_cast<size_t>(r * c) * 2;
      const int64_t B = std::min<int64_t>(64, std::max<int64_t>(1, (size_t(256) << 20) / per));
      const size_t need = per * B;
      if (need > have) {
        if (buf) cudaFree(buf);
        buf = nullptr;
        if (cudaMalloc(&buf, need) != cudaSuccess) {
          cudaGetLastError();
          st = MUON_ERR_OUT_OF_MEMORY;
          break;
        }
        have = need;
      }
      // a fixed, finite bf16 pattern (0x3c3c = 0.0115 in every element)
      if (cudaMemsetAsync(buf, 0x3c, need, stream) != cudaSuccess) {
        st = MUON_ERR_CUDA;
        break;
      }
      std::vector<float> t;
      for (int k = 0; k <= reps && st == MUON_OK; ++k) {   // run 0 warms up
        cudaEventRecord(e0, stream);
        st = ns_impl(buf, MUON_BF16, B, r, c, cfg, nullptr, stream);
        cudaEventRecord(e1, stream);
        if (st == MUON_OK && cudaEventSynchronize(e1) != cudaSuccess) st = MUON_ERR_CUDA;
        float ms = 0.f;
        if (st == MUON_OK && k > 0) {
          cudaEventElapsedTime(&ms, e0, e1);
          t.push_back(ms);
        }
      }
      if (st == MUON_OK) {
        std::sort(t.begin(), t.end());
        ms_per_matrix[i] = static_cast<double>(t[t.size() / 2]) / static_cast<double>(B);
      }
    }
    if (buf) {
      cudaStreamSynchronize(stream);
      cudaFree(buf);
    }
    cudaEventDestroy(e0);
    cudaEventDestroy(e1);
    return st;
  } catch (...) {
    return MUON_ERR_OUT_OF_MEMORY;
  }
}

muon_status_t muon_query_status(cudaStream_t stream) {
  try {
    std::lock_guard<std::mutex> lock(g_mu);
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_CUDA;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MUON_ERR_CUDA;
    // Two words may hold device-detected conditions: the one of the
    // allocating entry points (it exists once any of them ran here) and the
    // allocation-free entry point's, inside its fixed array.  Reading them
    // allocates nothing.
    unsigned v = 0;
    auto it = g_dev.find(dev);
    unsigned* words[2] = {it != g_dev.end() ? it->second.status : nullptr, noalloc_status_word(dev)};
    for (unsigned* w : words) {
      if (!w) continue;
      unsigned x = 0;
      if (cudaMemcpy(&x, w, sizeof(x), cudaMemcpyDeviceToHost) != cudaSuccess) return MUON_ERR_CUDA;
      if (x && cudaMemset(w, 0, sizeof(x)) != cudaSuccess) return MUON_ERR_CUDA;
      v |= x;
    }
    if (v) {
      for (auto& kv : g_ws) kv.second.dirty = true;
    }
    if (v & kDevBounds) return MUON_ERR_BOUNDS;
    if (v & kDevTimeout) return MUON_ERR_TIMEOUT;
    if (v & kDevNonfinite) return MUON_ERR_NONFINITE;
    return MUON_OK;
  } catch (...) {
    return MUON_ERR_CUDA;
  }
}

const char* muon_status_string(muon_status_t s) {
  switch (s) {
    case MUON_OK: return "MUON_OK";
    case MUON_ERR_INVALID_ARGUMENT: return "MUON_ERR_INVALID_ARGUMENT";
    case MUON_ERR_UNSUPPORTED: return "MUON_ERR_UNSUPPORTED";
    case MUON_ERR_ALIAS: return "MUON_ERR_ALIAS";
    case MUON_ERR_OUT_OF_MEMORY: return "MUON_ERR_OUT_OF_MEMORY";
    case MUON_ERR_CUDA: return "MUON_ERR_CUDA";
    case MUON_ERR_TIMEOUT: return "MUON_ERR_TIMEOUT";
    case MUON_ERR_NONFINITE: return "MUON_ERR_NONFINITE";
    case MUON_ERR_BOUNDS: return "MUON_ERR_BOUNDS";
    default: return "MUON_ERR_UNKNOWN";
  }
}

void muon_release_workspace(void) {
  try {
    std::lock_guard<std::mutex> lock(g_mu);
    int cur = 0;
    cudaGetDevice(&cur);
    for (auto& kv : g_ws) {
      if (kv.second.ptr || kv.second.ctr) {
        cudaSetDevice(kv.first.first);
        cudaStreamSynchronize(kv.first.second);
        if (kv.second.ptr) cudaFree(kv.second.ptr);
        if (kv.second.ctr) cudaFree(kv.second.ctr);
      }
    }
    g_ws.clear();
    for (auto& kv : g_host) {
      HostPipe& h = kv.second;
      cudaSetDevice(kv.first.first);
      for (cudaStream_t st : {h.s_in, h.s_comp, h.s_out})
        if (st) {
          cudaStreamSynchronize(st);
          cudaStreamDestroy(st);
        }
      if (h.ev_start) cudaEventDestroy(h.ev_start);
      for (int i = 0; i < kHostSlots; ++i)
        for (cudaEvent_t e : {h.ev_in[i], h.ev_comp[i], h.ev_free[i]})
          if (e) cudaEventDestroy(e);
      if (h.slot) cudaFree(h.slot);
    }
    g_host.clear();
    cudaSetDevice(cur);
  } catch (...) {
  }
}

int muon_last_launch_count(void) { return t_last_launches; }

int muon_ns_path(int64_t rows, int64_t cols, const muon_ns_config_t* cfg) {
  try {
    NsCfg ns;
    if (rows <= 0 || cols <= 0 || check_ns_cfg(cfg, &ns) != MUON_OK) return -1;
    const int64_t m = std::min(rows, cols), n = std::max(rows, cols);
    if (small_shape(m)) return 0;
    return gram_space_shape(m, n, ns) ? 2 : 1;
  } catch (...) {
    return -1;
  }
}

int muon_ns_gram_restart(int64_t m) { return m <= 0 ? -1 : gram_restart_period_env(m); }

int muon_debug_build(void) {
#ifdef MUON_DEBUG
  return 1;
#else
  return 0;
#endif
}

muon_status_t muon_debug_guard_check(cudaStream_t stream, int64_t* bad_bytes) {
  if (!bad_bytes) return MUON_ERR_INVALID_ARGUMENT;
  try {
    std::lock_guard<std::mutex> lock(g_mu);
    *bad_bytes = 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return MUON_ERR_CUDA;
    auto it = g_dev.find(dev);
    if (it == g_dev.end() || !it->second.guard_bad) return MUON_OK;
    if (cudaStreamSynchronize(stream) != cudaSuccess) return MUON_ERR_CUDA;
    unsigned long long v = 0;
    if (cudaMemcpy(&v, it->second.guard_bad, sizeof(v), cudaMemcpyDeviceToHost) != cudaSuccess)
      return MUON_ERR_CUDA;
    if (v && cudaMemset(it->second.guard_bad, 0, sizeof(v)) != cudaSuccess) return MUON_ERR_CUDA;
    *bad_bytes = static_cast<int64_t>(v);
    return MUON_OK;
  } catch (...) {
    return MUON_ERR_CUDA;
  }
}

muon_status_t muon_debug_inject_stall(int what) {
  if (what != 0 && what != kInjectGemm && what != kInjectSmall) return MUON_ERR_INVALID_ARGUMENT;
  g_inject.store(what);
  return MUON_OK;
}

int muon_profile_enable(int enable) {
  std::lock_guard<std::mutex> lock(g_mu);
  g_prof = enable != 0;
  return 7;
}

int muon_profile_read(double* ms, int64_t* launches, int n) {
  std::lock_guard<std::mutex> lock(g_mu);
  for (auto& r : g_prof_recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.e1) == cudaSuccess && cudaEventElapsedTime(&t, r.e0, r.e1) ==
                                                         cudaSuccess) {
      if (r.kind < n) {
        if (ms) ms[r.kind] += t;
        if (launches) launches[r.kind] += 1;
      }
    }
    cudaEventDestroy(r.e0);
    cudaEventDestroy(r.e1);
  }
  g_prof_recs.clear();
  return 7;
}

}  // extern "C"
