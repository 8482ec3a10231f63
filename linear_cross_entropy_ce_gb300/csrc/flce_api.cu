// C ABI of libflce: argument checks, workspace planning, TMA descriptors and
// the per-chunk launch sequence of the fused linear cross-entropy.
//
// Token-major chunking ("efficient-llm-anatomy" README, "Fused cross-entropy
// computes backward during forward": tokens are processed in chunks and each
// chunk runs all three matmuls).  For chunk c of C valid tokens:
//   gather   Xc = rows of X for the chunk's valid tokens
//   LOGITS   z = Xc W^T; per 128-column part max / sum-exp, target logit,
//            bf16 z - part max
//   lse_dz   lse per row (fixed-order merge), row loss, dz in place
//   BWD      one launch: DX grad_hidden rows = dz W (complete per chunk, K = V)
//            and DW grad_weight (+)= dz^T Xc (fixed chunk order, fp32)
// The only buffer that scales with V is the C x V bf16 chunk of logits, so
// the default plan keeps the workspace below 5% of the N x V bf16 logits.
#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <vector>

#include "flce.h"
#include "flce_internal.h"

namespace {

using namespace flce;

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(p);
  });
  return fn;
}

struct DeviceState {
  bool ready = false;
  int sms = 0;
  int major = 0;
  int pairs = 0;   // CTA pairs of the GEMM that fit on the device at once
};

constexpr int MAX_DEVICES = 64;
std::mutex g_dev_mu;
DeviceState g_dev[MAX_DEVICES];

cudaError_t device_state(DeviceState* out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= MAX_DEVICES) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_dev_mu);
  DeviceState& d = g_dev[dev];
  if (!d.ready) {
    if ((e = cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
    if ((e = cudaDeviceGetAttribute(&d.major, cudaDevAttrComputeCapabilityMajor, dev)) != cudaSuccess) return e;
    if ((e = gemm_prepare(dev)) != cudaSuccess) return e;
    if ((e = gemm_max_pairs(&d.pairs)) != cudaSuccess) return e;
    if (d.pairs < 1) return cudaErrorInvalidConfiguration;
    d.ready = true;
  }
  *out = d;
  return cudaSuccess;
}

unsigned long long wait_timeout_ns() {
  static unsigned long long v = [] {
    const char* s = std::getenv("FLCE_WAIT_TIMEOUT_NS");
    unsigned long long x = s ? std::strtoull(s, nullptr, 10) : 0ull;
    return x ? x : 2000000000ull;  // 2 s: far above any legitimate wait
  }();
  return v;
}

// ---------------------------------------------------------------------------
// workspace plan
// ---------------------------------------------------------------------------
struct Plan {
  long long N = 0, H = 0, V = 0, C = 0, ldz = 0, n_chunks = 0;
  int nvt = 0, nparts = 0, splits = 1, kb_per_split = 0;
  long long n_counters = 0, flags_per_chunk = 0;
  bool fwd_only = false, norm = false, gw32 = false;
  size_t o_idx = 0, o_rl = 0, o_cnt = 0, o_xc = 0, o_tc = 0, o_zt = 0, o_part = 0, o_z = 0, o_dx = 0, o_rinv = 0,
         o_dg = 0, o_gw = 0, total = 0;
};

inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }
inline long long cdiv(long long a, long long b) { return (a + b - 1) / b; }

constexpr int DEFAULT_PAIRS = 76;
constexpr int MAX_SPLITS = 16;   // splits are summed one after another: keep the chain short
constexpr int DX_UNIT_KB = 128;  // preferred K blocks of one dX unit

// Workspace layout for chunks of C rows.  Only the bf16 C x V logits buffer
// (absent for the forward-only call) grows with V; with a bf16 grad_weight
// (gw32) the fp32 V x H accumulator of grad_weight lives here as well.
Plan layout(long long N, long long H, long long V, long long C, int S, bool fwd_only, bool norm = false,
            bool gw32 = false) {
  Plan p;
  p.N = N; p.H = H; p.V = V; p.C = C; p.fwd_only = fwd_only; p.norm = norm; p.gw32 = gw32 && !fwd_only;
  p.ldz = cdiv(V, 64) * 64;
  p.nvt = static_cast<int>(cdiv(V, BN));
  p.nparts = static_cast<int>(cdiv(V, PART_COLS));
  p.n_chunks = cdiv(N, C);
  const long long kbt = cdiv(V, BK);
  if (fwd_only) S = 1;
  p.kb_per_split = static_cast<int>(cdiv(kbt, S));
  p.splits = static_cast<int>(cdiv(kbt, p.kb_per_split));
  p.flags_per_chunk = p.splits > 1 ? 4 * cdiv(C, PAIR_M) * cdiv(H, BN) : 0;   // (tile, CTA, warpgroup)
  p.n_counters = p.n_chunks * (2 + p.flags_per_chunk);   // tile counters, then split flags
  size_t off = al256(HDR_WORDS * sizeof(int));
  p.o_idx = off;  off += al256(size_t(N) * 4);
  p.o_rl = off;   off += al256(size_t(N) * 4);
  p.o_cnt = off;  off += al256(size_t(p.n_counters) * 4);
  p.o_xc = off;   off += al256(size_t(C) * H * 2);
  p.o_tc = off;   off += al256(size_t(C) * 4);
  p.o_zt = off;   off += al256(size_t(C) * 4);
  if (!fwd_only) { p.o_z = off; off += al256(size_t(C) * p.ldz * 2); }
  // The per-part (max, sum exp) of a chunk are read by lse_dz before the
  // backward launch, and the fp32 sum of a split grad_hidden GEMM lives only
  // inside that launch (the next chunk's logits rewrite the parts after it):
  // the two share their bytes.
  p.o_part = off;
  size_t shared = al256(size_t(C) * p.nparts * 8);
  if (!fwd_only && p.splits > 1) {
    p.o_dx = off;
    shared = std::max(shared, al256(size_t(C) * H * 4));
  }
  off += shared;
  if (norm) {   // final RMSNorm: 1/rms per chunk row, d(gain) partial per chunk
    p.o_rinv = off; off += al256(size_t(C) * 4);
    p.o_dg = off;   off += al256(size_t(p.n_chunks) * H * 4);
  }
  if (p.gw32) { p.o_gw = off; off += al256(size_t(V) * H * 4); }
  p.total = off;
  return p;
}

// Vocabulary splits of the grad_hidden GEMM.  A dX tile (K = V) should take at
// most a pair's average share of the backward launch, or it alone sets the
// launch's length (full-model shape: 2 splits 1.77 ms of backward per step,
// 4 splits 2.28 ms, 1 split 1.90 ms).  The parts of a tile are summed one after
// another, each waiting for the previous one to land (a few µs each), so the
// chain of S parts costs S of those steps unless the dX units are spread
// through the dW units (the kernel does that when the dW units outnumber what
// the other pairs need to stay busy during one dX unit).  Spread: short
// units (~DX_UNIT_KB K blocks) keep the spread even and the launch's tail
// short.  Not spread: S balances the unit length (kbt / S K blocks of
// ~0.3 µs) against the chain (S steps of ~4 µs), S ~ sqrt(kbt / 13).
int preferred_splits(long long C, long long H, long long V, int pairs) {
  const long long kbt = cdiv(V, BK);
  const double dx_tiles = double(cdiv(C, PAIR_M)) * double(cdiv(H, BN));
  const double unit = double(PAIR_M) * BN * double(V);
  const double work = dx_tiles * unit + double(cdiv(V, PAIR_M)) * double(cdiv(H, BN)) * PAIR_M * BN * double(C);
  const double per_pair = work / double(pairs);
  const long long balance = static_cast<long long>(std::ceil(unit / per_pair));
  const long long max_by_k = std::max<long long>(1, kbt / 8);   // >= 8 K blocks per split
  auto clamp = [&](long long S) {
    return std::max<long long>(1, std::min<long long>(std::min<long long>(S, MAX_SPLITS), max_by_k));
  };
  const long long n_dw = cdiv(V, PAIR_M) * cdiv(H, BN);
  const long long kb_dw = cdiv(C, BK);
  const long long spread = clamp(std::max<long long>(balance, cdiv(kbt, DX_UNIT_KB)));
  if (n_dw > static_cast<long long>(pairs) * cdiv(cdiv(kbt, spread), kb_dw)) return static_cast<int>(spread);
  const long long chain = std::llround(std::sqrt(double(kbt) / 13.0));
  return static_cast<int>(clamp(std::min<long long>(balance, chain)));
}

long long max_chunk(long long N) { return cdiv(N, BM) * BM; }

Plan plan_for_chunk(long long N, long long H, long long V, long long C, bool fwd_only, int pairs, size_t bytes,
                    bool norm = false, bool gw32 = false) {
  Plan p = layout(N, H, V, C, preferred_splits(C, H, V, pairs), fwd_only, norm, gw32);
  if (p.total > bytes) p = layout(N, H, V, C, 1, fwd_only, norm, gw32);
  return p;
}

// Largest chunk (multiple of 128 rows) whose plan fits in `bytes`.
bool plan_for_bytes(long long N, long long H, long long V, bool fwd_only, size_t bytes, int pairs, Plan* out,
                    bool norm = false, bool gw32 = false) {
  long long lo = BM, hi = max_chunk(N);
  if (layout(N, H, V, lo, 1, fwd_only, norm, gw32).total > bytes) return false;
  while (lo < hi) {   // the size shrinks as C grows only through the d(gain) partials: bisect on the total
    const long long mid = ((lo / BM + hi / BM + 1) / 2) * BM;
    if (layout(N, H, V, mid, 1, fwd_only, norm, gw32).total <= bytes) lo = mid;
    else hi = mid - BM;
  }
  *out = plan_for_chunk(N, H, V, lo, fwd_only, pairs, bytes, norm, gw32);
  return true;
}

int device_pairs() {
  DeviceState d;
  if (device_state(&d) == cudaSuccess) return d.pairs;
  cudaGetLastError();
  return DEFAULT_PAIRS;
}

bool sizes_ok(long long N, long long H, long long V) {
  return N >= 1 && H >= 8 && V >= 1 && N < (1ll << 31) && V < (1ll << 31) && H <= (1ll << 20) && H % 8 == 0;
}

// The default plan: chunk buffers within 5% of the bf16 logits (never below
// one 128-row chunk), plus the fp32 grad_weight accumulator when the caller
// asked for a bf16 grad_weight.
size_t default_bytes(long long N, long long H, long long V, bool fwd_only, bool norm = false, bool gw32 = false) {
  if (!sizes_ok(N, H, V)) return 0;
  gw32 = gw32 && !fwd_only;
  const size_t budget = size_t(N) * size_t(V) * 2 / 20 + (gw32 ? al256(size_t(V) * H * 4) : 0);
  const int pairs = device_pairs();
  Plan p;
  if (plan_for_bytes(N, H, V, fwd_only, budget, pairs, &p, norm, gw32)) return p.total;
  return plan_for_chunk(N, H, V, BM, fwd_only, pairs, ~size_t(0), norm, gw32).total;
}

constexpr uint32_t KNOWN_FLAGS = FLCE_REDUCE_SUM | FLCE_GW_BF16;

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

bool make_map(CUtensorMap* m, const void* base, unsigned long long inner, unsigned long long outer,
              unsigned long long row_bytes, unsigned box_inner, unsigned box_outer,
              CUtensorMapDataType dtype = CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
              CUtensorMapSwizzle swizzle = CU_TENSOR_MAP_SWIZZLE_128B) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  const cuuint64_t dims[2] = {inner, outer};
  const cuuint64_t strides[1] = {row_bytes};
  const cuuint32_t box[2] = {box_inner, box_outer};
  const cuuint32_t es[2] = {1, 1};
  return fn(m, dtype, 2, const_cast<void*>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// ---------------------------------------------------------------------------
// launch profiling (flce_profile_begin / flce_profile_end)
// ---------------------------------------------------------------------------
struct ProfRecord {
  int mode;
  cudaEvent_t start, stop;
};

struct Profiler {
  std::mutex mu;
  bool on = false;
  std::vector<cudaEvent_t> pool;  // events available for reuse
  std::vector<ProfRecord> recs;
  long long launches = 0;
};

Profiler& prof() {
  static Profiler p;
  return p;
}

cudaEvent_t prof_event() {
  Profiler& p = prof();
  if (!p.pool.empty()) {
    cudaEvent_t e = p.pool.back();
    p.pool.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  if (cudaEventCreate(&e) != cudaSuccess) { cudaGetLastError(); return nullptr; }
  return e;
}

// Test hook (flce_debug_arm_stall): a non-zero value arms the next GEMM
// launch of the process to withhold one pipeline signal, with this wait limit.
std::atomic<unsigned long long> g_stall_armed{0};

// Launch a GEMM, bracketed by events when profiling is on.
cudaError_t gemm_launch(const GemmArgs& g0, const GemmMaps& m, int grid, cudaStream_t st) {
  GemmArgs g = g0;
  if (const unsigned long long t = g_stall_armed.exchange(0)) {
    g.debug_stall = 1;
    g.timeout_ns = t;
  }
  Profiler& p = prof();
  std::unique_lock<std::mutex> lk(p.mu);
  if (!p.on) {
    lk.unlock();
    return launch_gemm(g, m, grid, st);
  }
  ProfRecord r{g.mode, prof_event(), prof_event()};
  if (r.start) cudaEventRecord(r.start, st);
  cudaError_t e = launch_gemm(g, m, grid, st);
  if (r.stop) cudaEventRecord(r.stop, st);
  if (r.start && r.stop) p.recs.push_back(r);
  ++p.launches;
  return e;
}

void count_launches(long long n) {
  Profiler& p = prof();
  std::lock_guard<std::mutex> lk(p.mu);
  if (p.on) p.launches += n;
}

template <typename T>
T* at(void* ws, size_t off) { return reinterpret_cast<T*>(static_cast<char*>(ws) + off); }

// One call of the library: the plain fused op, the forward-only loss, the
// fused final RMSNorm, or one of the two passes over a vocabulary shard.
enum JobKind { JOB_FWD_BWD, JOB_LOSS, JOB_SHARD_STATS, JOB_SHARD_BWD };

struct Job {
  JobKind kind = JOB_FWD_BWD;
  const void* hidden = nullptr;
  const void* weight = nullptr;      // the rows the GEMMs see: [V, H] (a shard: rows v0 .. v0+V-1)
  const int32_t* targets = nullptr;  // ids in the full vocabulary [0, V_total)
  int64_t N = 0, H = 0, V = 0, V_total = 0, v0 = 0;
  int32_t ii = -100;
  uint32_t flags = 0;
  float* loss = nullptr;
  int32_t* n_valid = nullptr;
  float* row_loss = nullptr;
  void* grad_hidden = nullptr;       // bf16 [N, H], or fp32 when grad_hidden_f32
  bool grad_hidden_f32 = false;
  float* grad_weight = nullptr;      // fp32 [V, H], or bf16 when FLCE_GW_BF16 is set
  const void* gain = nullptr;        // final RMSNorm
  float eps = 0.f;
  float* grad_gain = nullptr;
  float* row_max = nullptr;          // shard statistics
  float* row_sumexp = nullptr;
  float* row_zt = nullptr;
  const float* lse = nullptr;        // global log-sum-exp for the shard backward
  void* ws = nullptr;
  size_t ws_bytes = 0;
  void* stream = nullptr;
};

flce_status run(const Job& j) {
  const bool fwd_only = j.kind == JOB_LOSS || j.kind == JOB_SHARD_STATS;
  const bool norm = j.gain != nullptr;
  const int64_t N = j.N, H = j.H, V = j.V;
  if (norm && (!j.grad_gain || !aligned16(j.gain) || !aligned4(j.grad_gain) || !(j.eps >= 0.f))) return FLCE_EINVAL;
  if (!j.hidden || !j.weight || !j.targets || !j.ws) return FLCE_EINVAL;
  if ((j.kind == JOB_FWD_BWD || j.kind == JOB_LOSS) && (!j.loss || !j.n_valid)) return FLCE_EINVAL;
  if (!fwd_only && (!j.grad_hidden || !j.grad_weight)) return FLCE_EINVAL;
  if (j.kind == JOB_SHARD_STATS && (!j.row_max || !j.row_sumexp || !j.row_zt)) return FLCE_EINVAL;
  if (j.kind == JOB_SHARD_BWD && !j.lse) return FLCE_EINVAL;
  if (j.flags & ~KNOWN_FLAGS) return FLCE_EINVAL;
  const bool gw_bf16 = (j.flags & FLCE_GW_BF16) != 0;
  if (gw_bf16 && j.kind != JOB_FWD_BWD) return FLCE_EINVAL;   // forward-only and shard calls have no such output
  if (N < 1 || H < 1 || V < 1 || j.v0 < 0 || j.V_total < j.v0 + V) return FLCE_EINVAL;
  if (!sizes_ok(N, H, V) || j.V_total >= (1ll << 31)) return FLCE_EUNSUPPORTED;
  if (!aligned16(j.hidden) || !aligned16(j.weight) || !aligned16(j.ws) || !aligned4(j.targets) ||
      (j.loss && !aligned4(j.loss)) || (j.n_valid && !aligned4(j.n_valid)) || (j.row_loss && !aligned4(j.row_loss)))
    return FLCE_EUNSUPPORTED;
  if (!fwd_only && (!aligned16(j.grad_hidden) || !aligned16(j.grad_weight))) return FLCE_EUNSUPPORTED;
  if (j.lse && !aligned4(j.lse)) return FLCE_EUNSUPPORTED;

  DeviceState dev;
  if (device_state(&dev) != cudaSuccess) { cudaGetLastError(); return FLCE_ECUDA; }
  if (dev.major < 10) return FLCE_EUNSUPPORTED;
  Plan p;
  if (!plan_for_bytes(N, H, V, fwd_only, j.ws_bytes, dev.pairs, &p, norm, gw_bf16)) return FLCE_EWORKSPACE;

  cudaStream_t st = static_cast<cudaStream_t>(j.stream);
  void* ws = j.ws;
  int* hdr = at<int>(ws, 0);
  int* idx = at<int>(ws, p.o_idx);
  float* rl = at<float>(ws, p.o_rl);
  int* counters = at<int>(ws, p.o_cnt);
  uint16_t* xc = at<uint16_t>(ws, p.o_xc);
  int* tc = at<int>(ws, p.o_tc);
  float* zt = at<float>(ws, p.o_zt);
  float2* part = at<float2>(ws, p.o_part);
  uint16_t* z = fwd_only ? nullptr : at<uint16_t>(ws, p.o_z);
  float* dxacc = (!fwd_only && p.splits > 1) ? at<float>(ws, p.o_dx) : nullptr;
  float* rinv = norm ? at<float>(ws, p.o_rinv) : nullptr;
  float* dgp = norm ? at<float>(ws, p.o_dg) : nullptr;
  // the fp32 accumulator of grad_weight: the output itself, or a workspace
  // region that is rounded to the bf16 output at the end
  float* gwacc = p.gw32 ? at<float>(ws, p.o_gw) : j.grad_weight;

  GemmMaps fm, bm;   // forward (logits) and backward (dX + dW) launches
  std::memset(&fm, 0, sizeof(fm));
  std::memset(&bm, 0, sizeof(bm));
  const unsigned long long hb = static_cast<unsigned long long>(H) * 2;
  bool ok = make_map(&fm.a0, xc, H, p.C, hb, BK, BM) && make_map(&fm.b0, j.weight, H, V, hb, BK, BN / 2);
  if (!fwd_only)
    ok = ok && make_map(&bm.a0, z, V, p.C, p.ldz * 2, BK, BM) && make_map(&bm.b0, j.weight, H, V, hb, 64, BK) &&
         make_map(&bm.a1, z, V, p.C, p.ldz * 2, 64, BK) && make_map(&bm.b1, xc, H, p.C, hb, 64, BK) &&
         make_map(&bm.out, gwacc, H, V, static_cast<unsigned long long>(H) * 4, 32, 64,
                  CU_TENSOR_MAP_DATA_TYPE_FLOAT32, CU_TENSOR_MAP_SWIZZLE_128B);
  if (!ok) return FLCE_ECUDA;

  const int reduce_sum = (j.flags & FLCE_REDUCE_SUM) ? 1 : 0;
  GemmArgs g;
  std::memset(&g, 0, sizeof(g));
  g.hdr = hdr;
  g.status = hdr + HDR_STATUS;
  g.C = static_cast<int>(p.C);
  g.H = static_cast<int>(H);
  g.V = static_cast<int>(V);
  g.ldz = p.ldz;
  g.nvt = p.nvt;
  g.nparts = p.nparts;
  g.store_z = fwd_only ? 0 : 1;
  g.timeout_ns = wait_timeout_ns();
  g.z = z;
  g.part = part;
  g.zt = zt;
  g.tc = tc;
  g.idx = idx;
  g.grad_hidden = j.grad_hidden_f32 ? nullptr : static_cast<uint16_t*>(j.grad_hidden);
  g.grad_hidden_f32 = j.grad_hidden_f32 ? static_cast<float*>(j.grad_hidden) : nullptr;
  g.grad_weight = gwacc;
  g.splits = p.splits;
  g.kb_per_split = p.kb_per_split;
  g.interleave = 1;
  // grad_weight tiles of <= 8 K blocks are bound by their epilogue: the
  // epilogue threads pull the next grad_weight block into L2 with plain
  // prefetches (large-vocabulary workload, C = 384: the backward is 4% slower
  // without them).  Longer tiles prefetch nothing: a TMA prefetch of the block
  // at the tile start queued in front of the tile's loads and cost 0.6-2%
  // (Llama-3-8B head, full-model shape).
  g.pf_threads = p.C <= 512 ? 1 : 0;
  g.dxacc = dxacc;

  // persistent grids: CTA pairs, no more than fit on the device at once
  const long long mt = cdiv(p.C, PAIR_M), ht = cdiv(H, BN);
  const int grid_logits = 2 * static_cast<int>(std::min<long long>(mt * p.nvt, dev.pairs));
  const int grid_bwd =
      2 * static_cast<int>(std::min<long long>(mt * ht * p.splits + cdiv(V, PAIR_M) * ht, dev.pairs));

  auto chk = [](cudaError_t e) { return e == cudaSuccess; };
  const bool stats = j.kind == JOB_SHARD_STATS;
  const int v0 = static_cast<int>(j.v0);
  count_launches(1 + (fwd_only ? 0 : 1) + (j.kind == JOB_SHARD_BWD ? 0 : 1) + p.n_chunks * (norm ? 4 : 2) +
                 (norm ? 1 : 0) + (p.gw32 ? 1 : 0));
  if (!chk(launch_prep(j.targets, N, static_cast<int>(j.V_total), j.ii, hdr, idx, j.n_valid, counters,
                       p.n_counters, st)))
    return FLCE_ECUDA;
  if (!fwd_only && !chk(launch_zero_ignored(hdr, idx, N, H * (j.grad_hidden_f32 ? 4 : 2), j.grad_hidden, st)))
    return FLCE_ECUDA;
  if (stats && !chk(launch_shard_stats_ignored(hdr, idx, N, j.row_max, j.row_sumexp, j.row_zt, st)))
    return FLCE_ECUDA;
  for (long long c = 0; c < p.n_chunks; ++c) {
    const long long c0 = c * p.C;
    g.c0 = c0;
    if (norm) {
      if (!chk(launch_gather_norm(static_cast<const uint16_t*>(j.hidden), j.targets, hdr, idx, c0, g.C, g.H,
                                  static_cast<const uint16_t*>(j.gain), j.eps, xc, tc, rinv, st)))
        return FLCE_ECUDA;
    } else if (!chk(launch_gather(static_cast<const uint16_t*>(j.hidden), j.targets, hdr, idx, c0, g.C, g.H, xc,
                                  tc, v0, g.V, st))) {
      return FLCE_ECUDA;
    }
    int* sync = counters + c * (2 + p.flags_per_chunk);
    g.mode = MODE_LOGITS;
    g.counter = sync;
    if (!chk(gemm_launch(g, fm, grid_logits, st))) return FLCE_ECUDA;
    if (stats) {
      if (!chk(launch_shard_stats(hdr, idx, c0, g.C, p.nparts, part, zt, tc, j.row_max, j.row_sumexp, j.row_zt,
                                  st)))
        return FLCE_ECUDA;
      continue;
    }
    if (!chk(launch_lse_dz(hdr, c0, g.C, g.V, p.ldz, p.nparts, part, zt, tc, rl, z, reduce_sum, fwd_only ? 0 : 1,
                           j.lse, idx, st)))
      return FLCE_ECUDA;
    if (fwd_only) continue;
    g.mode = MODE_BWD;
    g.counter = sync + 1;
    g.flags = sync + 2;
    g.accumulate = c > 0 ? 1 : 0;
    g.first_chunk = c == 0 ? 1 : 0;
    if (!chk(gemm_launch(g, bm, grid_bwd, st))) return FLCE_ECUDA;
    if (norm && !chk(launch_rmsnorm_bwd(hdr, idx, c0, g.C, g.H, static_cast<const uint16_t*>(j.hidden),
                                        static_cast<const uint16_t*>(j.gain), rinv,
                                        static_cast<uint16_t*>(j.grad_hidden), dgp + c * H, st)))
      return FLCE_ECUDA;
  }
  if (j.kind == JOB_FWD_BWD || j.kind == JOB_LOSS) {
    if (!chk(launch_finalize(hdr, idx, rl, N, reduce_sum, j.loss, j.n_valid, j.row_loss, st))) return FLCE_ECUDA;
  }
  if (norm && !chk(launch_dgain_reduce(dgp, p.n_chunks, g.H, j.grad_gain, st))) return FLCE_ECUDA;
  if (p.gw32 && !chk(launch_f32_to_bf16(gwacc, V * H, reinterpret_cast<uint16_t*>(j.grad_weight), st)))
    return FLCE_ECUDA;
  return FLCE_OK;
}

flce_status run(const void* hidden, const void* weight, const int32_t* targets, int64_t N, int64_t H, int64_t V,
                int32_t ii, uint32_t flags, float* loss, int32_t* n_valid, float* row_loss, void* grad_hidden,
                float* grad_weight, void* ws, size_t ws_bytes, void* stream, bool fwd_only,
                const void* gain = nullptr, float eps = 0.f, float* grad_gain = nullptr) {
  Job j;
  j.kind = fwd_only ? JOB_LOSS : JOB_FWD_BWD;
  j.hidden = hidden; j.weight = weight; j.targets = targets;
  j.N = N; j.H = H; j.V = V; j.V_total = V; j.v0 = 0;
  j.ii = ii; j.flags = flags;
  j.loss = loss; j.n_valid = n_valid; j.row_loss = row_loss;
  j.grad_hidden = grad_hidden; j.grad_weight = grad_weight;
  j.gain = gain; j.eps = eps; j.grad_gain = grad_gain;
  j.ws = ws; j.ws_bytes = ws_bytes; j.stream = stream;
  return run(j);
}

}  // namespace

namespace flce {
// Forward+backward on a caller-provided device workspace (used by the entry
// point whose scratch is a static device array).
flce_status fwd_bwd_on_workspace(const void* hidden, const void* weight, const int32_t* targets, int64_t N,
                                 int64_t H, int64_t V, int32_t ignore_index, uint32_t flags, float* loss,
                                 int32_t* n_valid, float* row_loss, void* grad_hidden, float* grad_weight,
                                 void* workspace, size_t workspace_bytes, void* stream) {
  return run(hidden, weight, targets, N, H, V, ignore_index, flags, loss, n_valid, row_loss, grad_hidden,
             grad_weight, workspace, workspace_bytes, stream, false);
}
}  // namespace flce

extern "C" {

size_t flce_workspace_bytes(int64_t N, int64_t H, int64_t V, uint32_t flags) {
  if (flags & ~KNOWN_FLAGS) return 0;
  return default_bytes(N, H, V, false, false, (flags & FLCE_GW_BF16) != 0);
}

size_t flce_loss_workspace_bytes(int64_t N, int64_t H, int64_t V, uint32_t flags) {
  if (flags & ~FLCE_REDUCE_SUM) return 0;
  return default_bytes(N, H, V, true);
}

size_t flce_workspace_bytes_for_chunk(int64_t N, int64_t H, int64_t V, uint32_t flags, int64_t chunk_rows) {
  if ((flags & ~KNOWN_FLAGS) || !sizes_ok(N, H, V) || chunk_rows < 1) return 0;
  long long C = cdiv(chunk_rows, BM) * BM;
  if (C > max_chunk(N)) C = max_chunk(N);
  return plan_for_chunk(N, H, V, C, false, device_pairs(), ~size_t(0), false, (flags & FLCE_GW_BF16) != 0).total;
}

flce_status flce_plan(int64_t N, int64_t H, int64_t V, uint32_t flags, int forward_only, size_t workspace_bytes,
                      flce_plan_info* out) {
  if (!out || (flags & ~KNOWN_FLAGS)) return FLCE_EINVAL;
  if (N < 1 || H < 1 || V < 1) return FLCE_EINVAL;
  if (!sizes_ok(N, H, V)) return FLCE_EUNSUPPORTED;
  Plan p;
  if (!plan_for_bytes(N, H, V, forward_only != 0, workspace_bytes, device_pairs(), &p, false,
                      (flags & FLCE_GW_BF16) != 0))
    return FLCE_EWORKSPACE;
  out->chunk_rows = p.C;
  out->max_chunks = p.n_chunks;
  out->logits_row_stride = p.ldz;
  out->gemm_launches_per_chunk = forward_only ? 1 : 2;
  out->dx_splits = p.splits;
  out->vocab_tiles = p.nvt;
  out->workspace_bytes = p.total;
  return FLCE_OK;
}

flce_status flce_fwd_bwd(const void* hidden, const void* weight, const int32_t* targets, int64_t N, int64_t H,
                         int64_t V, int32_t ignore_index, uint32_t flags, float* loss, int32_t* n_valid,
                         float* row_loss, void* grad_hidden, float* grad_weight, void* workspace,
                         size_t workspace_bytes, void* stream) {
  return run(hidden, weight, targets, N, H, V, ignore_index, flags, loss, n_valid, row_loss, grad_hidden,
             grad_weight, workspace, workspace_bytes, stream, false);
}

flce_status flce_loss(const void* hidden, const void* weight, const int32_t* targets, int64_t N, int64_t H,
                      int64_t V, int32_t ignore_index, uint32_t flags, float* loss, int32_t* n_valid,
                      float* row_loss, void* workspace, size_t workspace_bytes, void* stream) {
  return run(hidden, weight, targets, N, H, V, ignore_index, flags, loss, n_valid, row_loss, nullptr, nullptr,
             workspace, workspace_bytes, stream, true);
}

flce_status flce_query_status(const void* workspace, void* stream) {
  if (!workspace || !aligned16(workspace)) return FLCE_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) { cudaGetLastError(); return FLCE_ECUDA; }
  int word = 0;
  if (cudaMemcpy(&word, static_cast<const int*>(workspace) + HDR_STATUS, sizeof(int), cudaMemcpyDeviceToHost) !=
      cudaSuccess) {
    cudaGetLastError();
    return FLCE_ECUDA;
  }
  if (word & STATUS_TIMEOUT) return FLCE_ETIMEOUT;
  if (word & STATUS_BADTARGET) return FLCE_EBADTARGET;
  return FLCE_OK;
}

flce_status flce_query_stall(const void* workspace, int32_t* info, void* stream) {
  if (!workspace || !aligned16(workspace) || !info) return FLCE_EINVAL;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) { cudaGetLastError(); return FLCE_ECUDA; }
  int w[2] = {0, 0};   // HDR_STALL, HDR_STALL_COUNT
  if (cudaMemcpy(w, static_cast<const int*>(workspace) + HDR_STALL, sizeof(w), cudaMemcpyDeviceToHost) !=
      cudaSuccess) {
    cudaGetLastError();
    return FLCE_ECUDA;
  }
  info[0] = w[0] & 0xff;
  info[1] = (w[0] >> 8) & 0xf;
  info[2] = w[0] >> 12;
  info[3] = w[1];
  return FLCE_OK;
}

flce_status flce_debug_arm_stall(uint64_t timeout_ns) {
  if (timeout_ns == 0 || timeout_ns > 10000000000ull) return FLCE_EINVAL;
  g_stall_armed.store(timeout_ns);
  return FLCE_OK;
}

size_t flce_rmsnorm_workspace_bytes(int64_t N, int64_t H, int64_t V, uint32_t flags) {
  if (flags & ~KNOWN_FLAGS) return 0;
  return default_bytes(N, H, V, false, true, (flags & FLCE_GW_BF16) != 0);
}

flce_status flce_rmsnorm_fwd_bwd(const void* hidden, const void* gain, float eps, const void* weight,
                                 const int32_t* targets, int64_t N, int64_t H, int64_t V, int32_t ignore_index,
                                 uint32_t flags, float* loss, int32_t* n_valid, float* row_loss, void* grad_hidden,
                                 float* grad_gain, float* grad_weight, void* workspace, size_t workspace_bytes,
                                 void* stream) {
  if (!gain || !grad_gain) return FLCE_EINVAL;
  return run(hidden, weight, targets, N, H, V, ignore_index, flags, loss, n_valid, row_loss, grad_hidden,
             grad_weight, workspace, workspace_bytes, stream, false, gain, eps, grad_gain);
}

size_t flce_vocab_shard_workspace_bytes(int64_t N, int64_t H, int64_t V_shard, uint32_t flags) {
  if (flags & ~FLCE_REDUCE_SUM) return 0;
  return default_bytes(N, H, V_shard, false);
}

flce_status flce_vocab_shard_stats(const void* hidden, const void* weight_shard, const int32_t* targets, int64_t N,
                                   int64_t H, int64_t V_shard, int64_t v0, int64_t V_total, int32_t ignore_index,
                                   float* row_max, float* row_sumexp, float* row_target_logit, int32_t* n_valid,
                                   void* workspace, size_t workspace_bytes, void* stream) {
  Job j;
  j.kind = JOB_SHARD_STATS;
  j.hidden = hidden; j.weight = weight_shard; j.targets = targets;
  j.N = N; j.H = H; j.V = V_shard; j.V_total = V_total; j.v0 = v0; j.ii = ignore_index;
  j.n_valid = n_valid;
  j.row_max = row_max; j.row_sumexp = row_sumexp; j.row_zt = row_target_logit;
  j.ws = workspace; j.ws_bytes = workspace_bytes; j.stream = stream;
  if (!row_max || !row_sumexp || !row_target_logit || !aligned4(row_max) || !aligned4(row_sumexp) ||
      !aligned4(row_target_logit))
    return FLCE_EINVAL;
  return run(j);
}

flce_status flce_vocab_rescale(const float* row_max_local, const float* row_max_global, float* row_sumexp,
                               int64_t N, void* stream) {
  if (!row_max_local || !row_max_global || !row_sumexp || N < 1) return FLCE_EINVAL;
  count_launches(1);
  return launch_vocab_rescale(row_max_local, row_max_global, row_sumexp, N, static_cast<cudaStream_t>(stream)) ==
                 cudaSuccess
             ? FLCE_OK
             : FLCE_ECUDA;
}

flce_status flce_vocab_finish(const float* row_max, const float* row_sumexp, const float* row_target_logit,
                              const int32_t* targets, int64_t N, int32_t ignore_index, uint32_t flags, float* lse,
                              float* row_loss, float* loss, int32_t* n_valid, void* stream) {
  if (!row_max || !row_sumexp || !row_target_logit || !targets || !loss || N < 1 || (flags & ~FLCE_REDUCE_SUM))
    return FLCE_EINVAL;
  count_launches(1);
  return launch_vocab_finish(row_max, row_sumexp, row_target_logit, targets, N, ignore_index,
                             (flags & FLCE_REDUCE_SUM) ? 1 : 0, lse, row_loss, loss, n_valid,
                             static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? FLCE_OK
             : FLCE_ECUDA;
}

flce_status flce_vocab_shard_bwd(const void* hidden, const void* weight_shard, const int32_t* targets, int64_t N,
                                 int64_t H, int64_t V_shard, int64_t v0, int64_t V_total, int32_t ignore_index,
                                 uint32_t flags, const float* lse, float* grad_hidden_partial,
                                 float* grad_weight_shard, void* workspace, size_t workspace_bytes, void* stream) {
  Job j;
  j.kind = JOB_SHARD_BWD;
  j.hidden = hidden; j.weight = weight_shard; j.targets = targets;
  j.N = N; j.H = H; j.V = V_shard; j.V_total = V_total; j.v0 = v0; j.ii = ignore_index; j.flags = flags;
  j.lse = lse;
  j.grad_hidden = grad_hidden_partial; j.grad_hidden_f32 = true;
  j.grad_weight = grad_weight_shard;
  j.ws = workspace; j.ws_bytes = workspace_bytes; j.stream = stream;
  return run(j);
}

flce_status flce_scale_grads(void* grad_hidden, float* grad_weight, int64_t N, int64_t H, int64_t V,
                             const float* scale, void* stream) {
  if (!grad_hidden || !grad_weight || !scale) return FLCE_EINVAL;
  if (N < 1 || H < 1 || V < 1) return FLCE_EINVAL;
  if (!sizes_ok(N, H, V)) return FLCE_EUNSUPPORTED;
  if (!aligned16(grad_hidden) || !aligned16(grad_weight) || !aligned4(scale)) return FLCE_EUNSUPPORTED;
  count_launches(1);
  if (launch_scale_grads(static_cast<uint16_t*>(grad_hidden), N * H, grad_weight, V * H, scale,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return FLCE_ECUDA;
  return FLCE_OK;
}

flce_status flce_selftest_timeout(void* workspace, uint64_t timeout_ns, void* stream) {
  if (!workspace || !aligned16(workspace) || timeout_ns == 0 || timeout_ns > 10000000000ull) return FLCE_EINVAL;
  if (launch_timeout_selftest(static_cast<int*>(workspace), timeout_ns, static_cast<cudaStream_t>(stream)) !=
      cudaSuccess)
    return FLCE_ECUDA;
  return FLCE_OK;
}

flce_status flce_profile_begin(void) {
  Profiler& p = prof();
  std::lock_guard<std::mutex> lk(p.mu);
  p.on = true;
  p.launches = 0;
  return FLCE_OK;
}

flce_status flce_profile_end(double* gemm_ms, int64_t* gemm_launches, int64_t* kernel_launches) {
  Profiler& p = prof();
  std::lock_guard<std::mutex> lk(p.mu);
  double ms[3] = {0, 0, 0};
  int64_t cnt[3] = {0, 0, 0};
  flce_status st = FLCE_OK;
  for (const ProfRecord& r : p.recs) {
    float t = 0.f;
    if (cudaEventSynchronize(r.stop) != cudaSuccess || cudaEventElapsedTime(&t, r.start, r.stop) != cudaSuccess) {
      cudaGetLastError();
      st = FLCE_ECUDA;
    } else if (r.mode >= 0 && r.mode < 3) {
      ms[r.mode] += t;
      ++cnt[r.mode];
    }
    p.pool.push_back(r.start);
    p.pool.push_back(r.stop);
  }
  p.recs.clear();
  for (int i = 0; i < 3; ++i) {
    if (gemm_ms) gemm_ms[i] = ms[i];
    if (gemm_launches) gemm_launches[i] = cnt[i];
  }
  if (kernel_launches) *kernel_launches = p.launches;
  p.on = false;
  p.launches = 0;
  return st;
}

const char* flce_status_string(flce_status s) {
  switch (s) {
    case FLCE_OK: return "ok";
    case FLCE_EINVAL: return "invalid argument";
    case FLCE_EUNSUPPORTED: return "unsupported size, alignment or device";
    case FLCE_EWORKSPACE: return "workspace too small";
    case FLCE_EBADTARGET: return "target outside [0, V) that is not ignore_index";
    case FLCE_ETIMEOUT: return "device pipeline wait timed out";
    case FLCE_ECUDA: return "CUDA error";
  }
  return "unknown status";
}

const char* flce_version(void) { return "0.1.0"; }

}  // extern "C"
