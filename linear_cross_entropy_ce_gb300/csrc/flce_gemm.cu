// Persistent tcgen05 GEMM with the epilogues of the fused linear
// cross-entropy ("efficient-llm-anatomy" README, "Fused cross-entropy
// computes backward during forward": per token chunk, logits = X W^T, then
// grad_input and grad_weight from the softmax of those logits).
//
//   MODE_LOGITS  z = Xc W^T           A = Xc [C,H] K-major,  B = W [V,H] K-major
//                epilogue: per row and 128-column vocabulary part the part
//                max m and sum exp(z - m) (one step of the online softmax of
//                "Alisa's book of LLMs", "Numerical stability and other
//                tricks"), the target logit, and z - m stored as bf16.
//   MODE_BWD     the two consumers of dz in one launch:
//     dX units   dX = dz W            A = dz [C,V] K-major,  B = W [V,H] MN-major
//                epilogue: bf16 rows of grad_hidden, scattered to token rows;
//                with the vocabulary split in S parts, the parts are summed in
//                fp32 in split order (a store, then L2 reduce-adds, each part
//                waiting for the previous one), and the last part converts.
//     dW units   dW (+)= dz^T Xc      A = dz^T (MN-major view of dz), B = Xc MN-major
//                epilogue: fp32 tile staged in shared memory, 64 x 32 boxes
//                of 128-byte rows, and written by a TMA store (first chunk)
//                or a TMA reduce-add (later chunks), so the fp32 accumulation
//                happens in L2 in fixed chunk order.
//                dX units are bound by the tensor cores, dW units (short, 12
//                K blocks at C = 768) by the latency of their loads under the
//                grad_weight read-modify-write: where the grad_hidden GEMM is
//                split, the claim order spreads the dX units evenly through
//                the dW units so both kinds run at once.
//
// Each tile is 256 x 256 and is computed by a CTA pair (a cluster of two CTAs
// on two SMs) with tcgen05.mma.cta_group::2: each CTA stages its 128 rows of
// A and its 128 columns of B (32 KB per K block) and holds 128 accumulator
// rows in its TMEM.  Per CTA: warp 0 issues TMA loads into a 6-stage ring (7
// in the logits launch, whose epilogue needs no staging buffers; in CTA 0 it
// also claims tiles from a global counter and hands them to both CTAs, to
// CTA 1 by st.async into a scheduler slot; slots and accumulators are handed
// back with relaxed arrives, since a release arrive waits for the thread's
// loads or stores in flight),
// warp 1 allocates TMEM and, in CTA 0, one lane issues the MMAs for the pair,
// and warps 2-17 are the epilogue: two sets of two warpgroups, set e draining
// TMEM accumulator e (double buffered, 2 x 256 columns), one 128-column half
// per warpgroup, so the epilogues of two consecutive tiles run at once and
// both overlap the next tile's main loop.  Every wait is bounded: on time-out
// a CTA raises an abort flag, lets copies in flight land, waits for its MMAs,
// frees TMEM and returns, and the workspace status word records
// STATUS_TIMEOUT.
#include "flce_internal.h"
#include "flce_ptx.cuh"

namespace flce {
namespace {

constexpr int STAGES = 6;                   // TMA ring of the backward launch
constexpr int STAGES_LOGITS = 7;            // the logits epilogue stages nothing: its ring also takes the staging area
constexpr int A_BYTES = BM * BK * 2;        // 16 KB: this CTA's 128 rows of A
constexpr int B_BYTES = (BN / 2) * BK * 2;  // 16 KB: this CTA's 128 columns of B
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int SLICE_COLS = 16;              // fp32 columns per staged slice of a split grad_hidden part (64 B rows)
// grad_weight leaves through TMA boxes of 64 rows x 32 fp32 columns (128-byte
// rows, 8 KB, one warpgroup's staging buffer); 128-byte rows halve the row
// requests of 64-byte ones
constexpr int OUT_COLS = 32;
constexpr int OUT_ROWS = 64;
constexpr int STG_BYTES = BM * SLICE_COLS * 4;   // a warpgroup's staging buffer: 8 KB
static_assert(OUT_ROWS * OUT_COLS * 4 == STG_BYTES, "one grad_weight box fills a staging buffer");
// Two epilogue sets, one per TMEM accumulator, so that the epilogues of two
// consecutive tiles run at once (tiles with few K blocks are bound by their
// epilogue); each set has two warpgroups, one per 128-column half.
constexpr int EPI_SETS = 2;
constexpr int SET_GROUPS = 2;
constexpr int EPI_GROUPS = EPI_SETS * SET_GROUPS;
constexpr int GROUP_COLS = BN / SET_GROUPS;
constexpr int GROUP_THREADS = 128;
constexpr int SET_THREADS = SET_GROUPS * GROUP_THREADS;
constexpr int EPI_THREADS = EPI_GROUPS * GROUP_THREADS;
constexpr int EPI_WARPS = EPI_THREADS / 32;
constexpr int NUM_THREADS = 64 + EPI_THREADS;   // warp 0 TMA, warp 1 MMA, then the epilogue warps
constexpr int SCHED_SLOTS = 4;
constexpr int SHORT_TILE_KB = 32;           // tiles with at most this many K blocks claim their successor early
constexpr uint32_t EPI_BAR_SET = 1;         // + set index: named barrier of one epilogue set
constexpr uint32_t EPI_BAR_GROUP = 1 + EPI_SETS;   // + warpgroup index: per-warpgroup named barrier
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int MN_BLOCK_BYTES = 64 * 128;    // 64 K rows x 128 B (64 bf16 along M or N)
constexpr uint16_t PAIR_MASK = 0x3;
constexpr float LOG2E = 1.4426950408889634f;

struct Ctl {
  uint64_t full[STAGES_LOGITS];  // CTA 0: both CTAs' loads of a stage landed
  uint64_t empty[STAGES_LOGITS]; // each CTA: the pair's MMAs released the stage
  uint64_t tfull[2];           // each CTA: accumulator ready
  uint64_t tempty[2];          // CTA 0: every warp of the accumulator's epilogue set in both CTAs has read it
  uint64_t sfull[SCHED_SLOTS]; // each CTA: a tile id is in sunit
  uint64_t sempty[SCHED_SLOTS];// CTA 0: every reader of the slot is done
  uint64_t mma_done;
  int sunit[SCHED_SLOTS];
  uint32_t tmem_base;
  int abort;
};

constexpr int CTL_BYTES = ((sizeof(Ctl) + 255) / 256) * 256;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + EPI_GROUPS * STG_BYTES + CTL_BYTES;   // one staging buffer per warpgroup
static_assert(SMEM_BYTES <= 232448, "shared memory budget");
static_assert(STAGES_LOGITS * STAGE_BYTES <= STAGES * STAGE_BYTES + EPI_GROUPS * STG_BYTES,
              "the extra logits stages fit in the epilogue staging area");

// Readers of a scheduler slot, one arrival per warp: in CTA 0 the MMA lane
// and the epilogue warps, in CTA 1 the TMA lane and the epilogue warps.
constexpr uint32_t SCHED_READERS = 2 * (1 + EPI_WARPS);
// Arrivals that free an accumulator: every warp of its set, in both CTAs.
constexpr uint32_t TEMPTY_ARRIVALS = 2 * (SET_THREADS / 32);

// Bounded wait on an mbarrier phase.  Gives up (returning false) when the
// CTA's abort flag is raised by another role, or after timeout_ns, in which
// case it raises the flag itself.
// Wait sites, recorded in the workspace header when a wait times out.
enum WaitSite : int {
  W_SCHED_EMPTY = 1, W_SCHED_FULL_PRODUCER = 2, W_STAGE_EMPTY = 3, W_DRAIN = 4, W_SCHED_FULL_MMA = 5,
  W_TMEM_EMPTY = 6, W_STAGE_FULL = 7, W_MMA_DONE = 8, W_SCHED_FULL_EPI = 9, W_TMEM_FULL = 10, W_SPLIT_FLAG = 11
};

// detail: the tile being worked on (or -1) and the ring position waited on
__device__ void record_stall(int* hdr, int site, int detail) {
  const int code = site | (static_cast<int>(ptx::cluster_ctarank()) << 8) | (static_cast<int>(blockIdx.x) << 12);
  atomicCAS(hdr + HDR_STALL, 0, code);
  const int k = atomicAdd(hdr + HDR_STALL_COUNT, 1);
  if (k < STALL_LOG_MAX) {
    hdr[HDR_STALL_LOG + 2 * k] = code;
    hdr[HDR_STALL_LOG + 2 * k + 1] = detail;
  }
}

__device__ __noinline__ bool wait_phase(uint64_t* bar, uint32_t parity, Ctl* ctl, uint64_t timeout_ns,
                                        bool honor_abort, int* hdr, int site, int detail = -1) {
  if (ptx::mbar_test_cluster(bar, parity)) return true;
  const uint64_t t0 = ptx::global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_test_cluster(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (honor_abort && *reinterpret_cast<volatile int*>(&ctl->abort)) return false;
      if (ptx::global_timer_ns() - t0 > timeout_ns) {
        *reinterpret_cast<volatile int*>(&ctl->abort) = 1;
        record_stall(hdr, site, detail);
        return false;
      }
    }
  }
}

// Wait on a stage barrier of the TMA ring (local, completed by TMA bytes or by
// the pair's MMA commit).  The common case, a phase that has already
// completed, costs one CTA-scope try_wait in line; the bounded cluster-scope
// loop above runs only when the phase is still open.  (Routing every stage
// wait through that loop cost the logits launch 6-8%.)
__device__ __forceinline__ bool wait_stage(uint64_t* bar, uint32_t parity, Ctl* ctl, uint64_t timeout_ns, int* hdr,
                                           int site, int detail) {
  if (ptx::mbar_test(bar, parity)) return true;
  return wait_phase(bar, parity, ctl, timeout_ns, true, hdr, site, detail);
}

// Bounded wait until a global flag reaches `target`.
__device__ __noinline__ bool wait_flag(const int* flag, int target, Ctl* ctl, uint64_t timeout_ns, int* hdr) {
  if (ptx::ld_acquire_gpu(flag) >= target) return true;
  const uint64_t t0 = ptx::global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ptx::ld_acquire_gpu(flag) >= target) return true;
    if ((i & 15u) == 0) {
      if (*reinterpret_cast<volatile int*>(&ctl->abort)) return false;
      if (ptx::global_timer_ns() - t0 > timeout_ns) {
        *reinterpret_cast<volatile int*>(&ctl->abort) = 1;
        record_stall(hdr, W_SPLIT_FLAG, target);
        return false;
      }
    }
    __nanosleep(64);
  }
}

struct Shape {
  int Cl;         // valid rows in this chunk
  int mt, nt;     // LOGITS: pair tiles along M and N; BWD: dX pair tiles along M and N
  int kbt;        // LOGITS: K blocks
  int n_dx;       // BWD: number of dX units
  int dw_mt;      // BWD: dW pair tiles along M (vocabulary)
  int dx_span;    // BWD: the dX units are spread over claim positions [0, dx_span)
  int units;
};

__device__ __forceinline__ Shape make_shape(const GemmArgs& a) {
  Shape s;
  const long long nv = a.hdr[HDR_NVALID];
  const long long rem = nv - a.c0;
  s.Cl = rem <= 0 ? 0 : (rem >= a.C ? a.C : static_cast<int>(rem));
  s.mt = (s.Cl + PAIR_M - 1) / PAIR_M;
  if (a.mode == MODE_LOGITS) {
    s.nt = a.nvt;
    s.kbt = (a.H + BK - 1) / BK;
    s.n_dx = 0;
    s.dw_mt = 0;
    s.dx_span = 0;
    s.units = s.mt * s.nt;
  } else {
    s.nt = (a.H + BN - 1) / BN;
    s.kbt = 0;
    s.n_dx = s.mt * s.nt * a.splits;
    s.dw_mt = (a.V + PAIR_M - 1) / PAIR_M;
    const int n_dw = s.dw_mt * s.nt;
    s.units = s.Cl > 0 ? s.n_dx + n_dw : 0;
    s.dx_span = s.n_dx;   // dX units first
    if (a.interleave && s.Cl > 0) {
      // Leave after the last dX unit enough dW units for every other pair to
      // stay busy while it runs: about one dX unit of work per pair.
      const long long kb_dw = (s.Cl + BK - 1) / BK;
      const long long tail =
          min(static_cast<long long>(n_dw), static_cast<long long>(gridDim.x / 2) * ((a.kb_per_split + kb_dw - 1) / kb_dw));
      s.dx_span = s.n_dx + n_dw - static_cast<int>(tail);
    }
  }
  return s;
}

enum UnitKind : int { U_LOGITS = 0, U_DX = 1, U_DW = 2 };

struct Unit {
  int kind;
  int m0, n0;     // pair tile origin (rows of the pair, columns)
  int ntile;      // vocab tile (LOGITS), dX tile index (DX)
  int split;      // DX vocabulary split
  int kb0, kb1;
};

// Tile order: LOGITS walks M fastest so the pairs in flight share one W tile.
// BWD: claim position u holds a dX unit when ceil(u n_dx / dx_span) steps up
// at u (dX units evenly spread over [0, dx_span), the first at u = 0), else
// the next dW unit.  dX units walk M fastest, so the units claimed close
// together share one slice of W; then N; then the vocabulary split, so every
// split is claimed after the previous one of its tile.  dW units walk N
// fastest so they share one slab of dz.
__device__ __forceinline__ Unit decode_unit(const GemmArgs& a, const Shape& s, int u) {
  Unit t;
  t.split = 0;
  if (a.mode == MODE_LOGITS) {
    const int m = u % s.mt, n = u / s.mt;
    t.kind = U_LOGITS; t.m0 = m * PAIR_M; t.n0 = n * BN; t.ntile = n; t.kb0 = 0; t.kb1 = s.kbt;
    return t;
  }
  int dx_before = s.n_dx;   // dX units at positions below u
  bool is_dx = false;
  if (u < s.dx_span) {
    const long long span = s.dx_span;
    dx_before = static_cast<int>((static_cast<long long>(u) * s.n_dx + span - 1) / span);
    is_dx = static_cast<int>((static_cast<long long>(u + 1) * s.n_dx + span - 1) / span) > dx_before;
  }
  if (is_dx) {
    const int i = dx_before;
    const int m = i % s.mt, rest = i / s.mt;
    const int n = rest % s.nt, sp = rest / s.nt;
    const int kbt = (a.V + BK - 1) / BK;
    t.kind = U_DX; t.m0 = m * PAIR_M; t.n0 = n * BN; t.ntile = m * s.nt + n; t.split = sp;
    t.kb0 = sp * a.kb_per_split;
    t.kb1 = min(kbt, t.kb0 + a.kb_per_split);
  } else {
    const int w = u - dx_before;
    const int n = w % s.nt, m = w / s.nt;
    t.kind = U_DW; t.m0 = m * PAIR_M; t.n0 = n * BN; t.ntile = n; t.kb0 = 0; t.kb1 = (s.Cl + BK - 1) / BK;
  }
  return t;
}

// ---------------------------------------------------------------------------
// epilogues: one thread = one accumulator row of this CTA; each warpgroup owns
// 128 of the 256 columns.  tbase = this warp's TMEM lanes at the warpgroup's
// first column; row0 = first row of this CTA's half of the pair tile; col0 =
// first column of the warpgroup inside the tile.
// ---------------------------------------------------------------------------

__device__ __forceinline__ void epi_logits(const GemmArgs& a, const Shape& s, const Unit& t, int row0, int col0,
                                           uint32_t tbase, int r) {
  const int grow = row0 + r;
  const bool rv = grow < s.Cl;
  const int c0 = t.n0 + col0;                     // first vocabulary column of this part
  const int tgt = rv ? a.tc[grow] : -1;
  const int tl = tgt - c0;
  const int ncol = min(GROUP_COLS, a.V - c0);     // may be <= 0 past the vocabulary
  if (ncol <= 0) return;                          // uniform over the warpgroup
  float mx = -INFINITY, ztv = 0.f;
#pragma unroll 1
  for (int j = 0; j < GROUP_COLS / 32; ++j) {
    float v[32];
    ptx::tmem_ld32(tbase + j * 32, v);
    if (j * 32 + 32 <= ncol) {   // whole block inside the vocabulary
#pragma unroll
      for (int k = 0; k < 32; ++k) mx = fmaxf(mx, v[k]);
    } else {
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (j * 32 + k < ncol) mx = fmaxf(mx, v[k]);
    }
    if (static_cast<unsigned>(tl - j * 32) < 32u) {   // this row's target is in the block
#pragma unroll
      for (int k = 0; k < 32; ++k)
        if (j * 32 + k == tl) ztv = v[k];
    }
  }
  float sum = 0.f;
  uint16_t* zrow = a.z + static_cast<size_t>(grow) * a.ldz + c0;
  const bool store = a.store_z && rv;
  const float mb = -mx * LOG2E;
#pragma unroll 1
  for (int j = 0; j < GROUP_COLS / 32; ++j) {
    float v[32];
    ptx::tmem_ld32(tbase + j * 32, v);
    uint32_t pk[16];
    if (j * 32 + 32 <= ncol) {   // whole block inside the vocabulary
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        sum += ptx::ex2(fmaf(v[k], LOG2E, mb)) + ptx::ex2(fmaf(v[k + 1], LOG2E, mb));
        pk[k / 2] = ptx::pack_bf16x2(v[k] - mx, v[k + 1] - mx);
      }
    } else {
#pragma unroll
      for (int k = 0; k < 32; k += 2) {
        const int c = j * 32 + k;
        if (c < ncol) sum += ptx::ex2(fmaf(v[k], LOG2E, mb));
        if (c + 1 < ncol) sum += ptx::ex2(fmaf(v[k + 1], LOG2E, mb));
        pk[k / 2] = ptx::pack_bf16x2(v[k] - mx, v[k + 1] - mx);
      }
    }
    if (store && c0 + j * 32 < a.ldz) {   // 64 bytes of this row: two 32-byte stores
      uint16_t* dst = zrow + j * 32;
      ptx::st_global_v8(dst, pk[0], pk[1], pk[2], pk[3], pk[4], pk[5], pk[6], pk[7]);
      ptx::st_global_v8(dst + 16, pk[8], pk[9], pk[10], pk[11], pk[12], pk[13], pk[14], pk[15]);
    }
  }
  if (rv) {
    a.part[static_cast<size_t>(grow) * a.nparts + c0 / PART_COLS] = make_float2(mx, sum);
    if (tl >= 0 && tl < ncol) a.zt[grow] = ztv;
  }
}

__device__ __forceinline__ void store_bf16_row(uint16_t* dst, const float* v, int h, int H) {
#pragma unroll
  for (int g = 0; g < 4; ++g) {
    if (h + g * 8 < H) {
      const float* q = v + 8 * g;
      *reinterpret_cast<uint4*>(dst + 8 * g) =
          make_uint4(ptx::pack_bf16x2(q[0], q[1]), ptx::pack_bf16x2(q[2], q[3]), ptx::pack_bf16x2(q[4], q[5]),
                     ptx::pack_bf16x2(q[6], q[7]));
    }
  }
}

__device__ __forceinline__ void store_f32_row(float* dst, const float* v, int h, int H) {
#pragma unroll
  for (int g = 0; g < 8; ++g)
    if (h + g * 4 < H)
      *reinterpret_cast<float4*>(dst + 4 * g) = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
}

__device__ __forceinline__ void epi_dx_direct(const GemmArgs& a, const Shape& s, const Unit& t, int row0, int col0,
                                              uint32_t tbase, int r) {
  const int grow = row0 + r;
  const bool rv = grow < s.Cl;
  const long long tok = rv ? a.idx[a.c0 + grow] : 0;
#pragma unroll 1
  for (int j = 0; j < GROUP_COLS / 32; ++j) {
    const int h = t.n0 + col0 + j * 32;
    if (h >= a.H) break;  // warp-uniform
    float v[32];
    ptx::tmem_ld32(tbase + j * 32, v);
    if (!rv) continue;
    if (a.grad_hidden_f32) store_f32_row(a.grad_hidden_f32 + tok * a.H + h, v, h, a.H);
    else store_bf16_row(a.grad_hidden + tok * a.H + h, v, h, a.H);
  }
}

// The warpgroup's 128 x 128 fp32 accumulator block -> 32-column slices, each
// in two boxes of 64 rows -> shared memory (128-byte rows, 128-byte swizzle:
// chunk g of row rr sits at g ^ (rr & 7)) -> TMA store (reduce == false) or
// TMA reduce-add into `map` at (h, row0 + 64 b).  One 8 KB staging buffer per
// warpgroup (the four warpgroups keep the TMA unit busy between them), which
// the two row halves take in turn; `leader` (one thread of the warpgroup)
// owns the bulk groups.
__device__ __forceinline__ void block_to_global(const CUtensorMap* map, int ncols_total, int h0, int row0,
                                                bool reduce, uint32_t tbase, int r, bool leader, uint32_t bar,
                                                uint8_t* buf) {
  const int left = ncols_total - h0;
  const int nsl = left <= 0 ? 0 : min(GROUP_COLS / OUT_COLS, (left + OUT_COLS - 1) / OUT_COLS);
  if (nsl == 0) return;   // uniform over the warpgroup
  const int half = r / OUT_ROWS, rr = r % OUT_ROWS;   // the box (64 rows) this thread's row goes in
  uint8_t* row = buf + rr * (OUT_COLS * 4);
#pragma unroll 1
  for (int j = 0; j < nsl; ++j) {
    float v[OUT_COLS];
    ptx::tmem_ld32(tbase + j * OUT_COLS, v);
    const int h = h0 + j * OUT_COLS;
#pragma unroll 1
    for (int b = 0; b < BM / OUT_ROWS; ++b) {
      if (leader) ptx::bulk_wait_read_0();          // the previous box's store has read the buffer
      ptx::named_bar_sync(bar, GROUP_THREADS);
      if (half == b) {
#pragma unroll
        for (int g = 0; g < OUT_COLS / 4; ++g)      // 128-byte swizzle: 16-byte chunk g of row rr
          *reinterpret_cast<float4*>(row + ((g ^ (rr & 7)) << 4)) =
              make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
        ptx::fence_proxy_async_smem();
      }
      ptx::named_bar_sync(bar, GROUP_THREADS);
      if (leader) {
        if (reduce)
          ptx::tma_reduce_add_2d(map, buf, h, row0 + b * OUT_ROWS);
        else
          ptx::tma_store_2d(map, buf, h, row0 + b * OUT_ROWS);
        ptx::bulk_commit();
      }
    }
  }
}

// One warp's 32 accumulator rows x 128 fp32 columns -> dst rows [row0,
// row0 + 32), columns [h0, h0 + 128) of a [rows][ncols] fp32 array, 16
// columns at a time: a tcgen05 load gives each thread one row, the slice is
// turned around in the warp's own 2 KB of shared memory (64-byte rows,
// 16-byte chunks swizzled so that the row writes and the transposed reads are
// both conflict-free), and each vector access of the warp then covers 8 rows
// x 64 contiguous bytes: st.global.v4 (store) or red.global.add.v4.f32
// (accumulate, performed at L2).  For one SM alone this moves the block
// about twice as fast as TMA stores or reduce-adds of 16 x 128 boxes, which
// is what the ordered chain of grad_hidden splits needs; with every SM
// updating grad_weight at once the TMA reduce-add is faster (the
// Llama-3-8B-head backward is 9% slower with this path), so grad_weight
// keeps block_to_global.  Rows >= nrows and columns >= ncols are skipped.
__device__ __forceinline__ void warp_block_to_global(float* dst, int nrows, int ncols, int h0, int row0, bool reduce,
                                                     uint32_t tbase, int lane, uint8_t* wbuf) {
  const int left = ncols - h0;
  const int nsl = left <= 0 ? 0 : min(GROUP_COLS / SLICE_COLS, (left + SLICE_COLS - 1) / SLICE_COLS);
  uint8_t* wrow = wbuf + lane * (SLICE_COLS * 4);
  const int wsw = (lane >> 1) & 3;
  const int c = lane & 3;                   // the 16-byte chunk this thread moves
#pragma unroll 1
  for (int j = 0; j < nsl; ++j) {           // uniform over the warp
    float v[SLICE_COLS];
    ptx::tmem_ld16(tbase + j * SLICE_COLS, v);
#pragma unroll
    for (int g = 0; g < 4; ++g)
      *reinterpret_cast<float4*>(wrow + ((g ^ wsw) << 4)) = make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
    __syncwarp();
    const int h = h0 + j * SLICE_COLS + 4 * c;
#pragma unroll
    for (int p = 0; p < 4; ++p) {
      const int rr = (lane >> 2) + 8 * p;
      const float4 x = *reinterpret_cast<const float4*>(wbuf + rr * (SLICE_COLS * 4) + ((c ^ ((rr >> 1) & 3)) << 4));
      if (row0 + rr < nrows && h < ncols) {
        float* d = dst + static_cast<size_t>(row0 + rr) * ncols + h;
        if (reduce)
          ptx::red_add_v4(d, x);
        else
          *reinterpret_cast<float4*>(d) = x;
      }
    }
    __syncwarp();
  }
}

// dX unit of a split vocabulary: split 0 stores its fp32 part, split k waits
// until split k-1 has landed and reduce-adds onto it, the last split turns
// the finished fp32 rows into bf16 grad_hidden rows.  Each warpgroup orders
// its own column half.  Returns false on abort.
__device__ __forceinline__ bool epi_dx_split(const GemmArgs& a, const Shape& s, const Unit& t, int row0, int col0,
                                             int half_idx, uint32_t rank, uint32_t tbase, int r, int q, int lane,
                                             bool leader, uint32_t bar, uint8_t* wbuf, Ctl* ctl) {
  int* flag = a.flags + 4 * t.ntile + 2 * static_cast<int>(rank) + half_idx;
  bool ok = true;
  if (leader && t.split > 0) ok = wait_flag(flag, t.split, ctl, a.timeout_ns, const_cast<int*>(a.hdr));
  if (!ptx::named_bar_and(bar, GROUP_THREADS, ok)) return false;
  const int h0 = t.n0 + col0;
  float* acc = const_cast<float*>(a.dxacc);
  warp_block_to_global(acc, a.C, a.H, h0, row0 + q * 32, t.split > 0, tbase, lane, wbuf);
  __threadfence();                          // this part is in global memory before the flag moves on
  ptx::named_bar_sync(bar, GROUP_THREADS);
  if (leader) ptx::st_release_gpu(flag, t.split + 1);
  if (t.split == a.splits - 1) {
    const int grow = row0 + r;
    if (grow < s.Cl) {
      const long long tok = a.idx[a.c0 + grow];
      const float* src = a.dxacc + static_cast<size_t>(grow) * a.H;
      for (int j = 0; j < GROUP_COLS / 32; ++j) {
        const int h = h0 + j * 32;
        if (h >= a.H) break;
        float v[32];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          if (h + 4 * g < a.H) {
            const float4 x = __ldcg(reinterpret_cast<const float4*>(src + h + 4 * g));
            v[4 * g] = x.x; v[4 * g + 1] = x.y; v[4 * g + 2] = x.z; v[4 * g + 3] = x.w;
          } else {
            v[4 * g] = v[4 * g + 1] = v[4 * g + 2] = v[4 * g + 3] = 0.f;
          }
        }
        if (a.grad_hidden_f32) store_f32_row(a.grad_hidden_f32 + tok * a.H + h, v, h, a.H);
        else store_bf16_row(a.grad_hidden + tok * a.H + h, v, h, a.H);
      }
    }
  }
  return true;
}

__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(NUM_THREADS, 1)
    flce_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stg = smem + STAGES * STAGE_BYTES;
  Ctl* ctl = reinterpret_cast<Ctl*>(stg + EPI_GROUPS * STG_BYTES);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;
  const uint32_t rank = ptx::cluster_ctarank();
  const bool lead = rank == 0;

  const Shape s = make_shape(a);   // identical in both CTAs of a pair
  if (a.mode == MODE_BWD && s.Cl == 0) {
    // Empty first chunk (no valid token at all): grad_weight is zero.
    if (a.first_chunk) {
      const size_t n4 = static_cast<size_t>(a.V) * a.H / 4;
      float4* gw = reinterpret_cast<float4*>(a.grad_weight);
      for (size_t i = static_cast<size_t>(blockIdx.x) * NUM_THREADS + threadIdx.x; i < n4;
           i += static_cast<size_t>(gridDim.x) * NUM_THREADS)
        gw[i] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    return;
  }
  if (s.units == 0) return;

  if (threadIdx.x == 0) {
    for (int i = 0; i < STAGES_LOGITS; ++i) {
      ptx::mbar_init(&ctl->full[i], 1);
      ptx::mbar_init(&ctl->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&ctl->tfull[i], 1);
      ptx::mbar_init(&ctl->tempty[i], TEMPTY_ARRIVALS);
    }
    for (int i = 0; i < SCHED_SLOTS; ++i) {
      ptx::mbar_init(&ctl->sfull[i], 1);
      ptx::mbar_init(&ctl->sempty[i], SCHED_READERS);
      // CTA 1's slots are filled by CTA 0's st.async: its producer arms each
      // phase with the 4 bytes to expect (this one, then after each read)
      if (rank == 1) ptx::mbar_arrive_expect_tx(&ctl->sfull[i], 4);
    }
    ptx::mbar_init(&ctl->mma_done, 1);
    ctl->abort = 0;
    ptx::mbar_fence_init();
    ptx::tma_prefetch_desc(&maps.a0);
    ptx::tma_prefetch_desc(&maps.b0);
    if (a.mode == MODE_BWD) {
      ptx::tma_prefetch_desc(&maps.a1);
      ptx::tma_prefetch_desc(&maps.b1);
      ptx::tma_prefetch_desc(&maps.out);
    }
  }
  if (warp == 1) {
    ptx::tmem_alloc_pair(&ctl->tmem_base, TMEM_COLS);   // collective over the pair
    ptx::tmem_relinquish_pair();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::cluster_sync();   // both CTAs' barriers exist before any remote arrive
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const uint64_t to = a.timeout_ns;
  int* hdr = const_cast<int*>(a.hdr);
  const int half = static_cast<int>(rank) * BM;   // this CTA's rows (A) / columns (B) inside a pair tile
  const uint32_t nstages = a.mode == MODE_LOGITS ? STAGES_LOGITS : STAGES;

  if (warp == 0 && lane == 0) {
    // ---------------- (CTA 0: scheduler +) TMA producer ----------------
    uint32_t stage = 0, phase = 0, sslot = 0, sphase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;
    const uint32_t full0 = ptx::map_to_rank(&ctl->full[0], 0);       // the stage barriers are contiguous
    bool ok = true;
    // CTA 0 claims tiles from the global counter.  After a short tile the
    // claim latency would stall the ring between tiles, so the next tile is
    // claimed as soon as a short tile starts (its loads hide the atomic); a
    // long tile claims its successor only when its own loads are all issued,
    // so that it never holds work another pair could start.
    int next = lead ? atomicAdd(a.counter, 1) : -1;
    for (;;) {
      int u;
      if (lead) {
        if (!wait_phase(&ctl->sempty[sslot], sphase ^ 1u, ctl, to, true, hdr, W_SCHED_EMPTY)) { ok = false; break; }
        if (next < 0) next = atomicAdd(a.counter, 1);
        u = next < s.units ? next : -1;
        next = -1;
        ctl->sunit[sslot] = u;
        ptx::mbar_arrive(&ctl->sfull[sslot]);
        // the peer's copy goes by st.async, which completes the transaction
        // armed on the peer's slot barrier; a release arrive here would wait
        // for this thread's TMA loads in flight (~1 us per grad_weight tile)
        ptx::st_async_u32(ptx::map_to_rank(&ctl->sunit[sslot], 1), static_cast<uint32_t>(u),
                          ptx::map_to_rank(&ctl->sfull[sslot], 1));
      } else {
        if (!wait_phase(&ctl->sfull[sslot], sphase, ctl, to, true, hdr, W_SCHED_FULL_PRODUCER)) { ok = false; break; }
        u = ptx::ld_acquire_shared(&ctl->sunit[sslot]);
        ptx::mbar_arrive_expect_tx(&ctl->sfull[sslot], 4);   // arm the slot's next phase
        // hand the slot back; relaxed (the acquire load above orders it after
        // the read), since a release would wait for this thread's TMA loads
        ptx::mbar_arrive_remote_relaxed(ptx::map_to_rank(&ctl->sempty[sslot], 0));
      }
      if (++sslot == SCHED_SLOTS) { sslot = 0; sphase ^= 1u; }
      if (u < 0) break;
      const Unit t = decode_unit(a, s, u);
      if (lead && t.kb1 - t.kb0 <= SHORT_TILE_KB) next = atomicAdd(a.counter, 1);
      for (int kb = t.kb0; kb < t.kb1; ++kb) {
        if (!wait_stage(&ctl->empty[stage], phase ^ 1u, ctl, to, hdr, W_STAGE_EMPTY, u | (stage << 24))) { ok = false; break; }
        uint8_t* sa = smem + stage * STAGE_BYTES;
        uint8_t* sb = sa + A_BYTES;
        const uint32_t fb = full0 + stage * 8u;                        // CTA 0's barrier of this stage
        if (lead) ptx::mbar_arrive_expect_tx(&ctl->full[stage], 2 * STAGE_BYTES);
        const int k0 = kb * BK;
        if (t.kind == U_LOGITS) {
          ptx::tma_load_2d_pair(sa, &maps.a0, fb, k0, t.m0 + half);      // Xc rows, cols k0..
          ptx::tma_load_2d_pair(sb, &maps.b0, fb, k0, t.n0 + half);      // W rows (vocab), cols k0..
        } else if (t.kind == U_DX) {
          ptx::tma_load_2d_pair(sa, &maps.a0, fb, k0, t.m0 + half);      // dz rows, vocab k0..
#pragma unroll
          for (int j = 0; j < BN / 128; ++j)                              // W rows k0.., cols n0+half+64j
            ptx::tma_load_2d_pair(sb + j * MN_BLOCK_BYTES, &maps.b0, fb, t.n0 + half + 64 * j, k0);
        } else {
#pragma unroll
          for (int j = 0; j < BM / 64; ++j)                               // dz rows k0.., vocab m0+half+64j
            ptx::tma_load_2d_pair(sa + j * MN_BLOCK_BYTES, &maps.a1, fb, t.m0 + half + 64 * j, k0);
#pragma unroll
          for (int j = 0; j < BN / 128; ++j)                              // Xc rows k0.., cols n0+half+64j
            ptx::tma_load_2d_pair(sb + j * MN_BLOCK_BYTES, &maps.b1, fb, t.n0 + half + 64 * j, k0);
        }
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == nstages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
    if (!ok && lead) {
      // let the copies already in flight land before the pair exits
      for (int i = 0; i < nstages; ++i)
        if (issued_mask & (1u << i)) wait_phase(&ctl->full[i], (issued_parity >> i) & 1u, ctl, to, false, hdr, W_DRAIN);
    }
  } else if (warp == 1 && lane == 0 && lead) {
    // ---------------- MMA issuer for the pair ----------------
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, sslot = 0, sphase = 0;
    bool withhold = a.debug_stall != 0;   // test hook, see GemmArgs::debug_stall
    for (;;) {
      if (!wait_phase(&ctl->sfull[sslot], sphase, ctl, to, true, hdr, W_SCHED_FULL_MMA)) break;
      const int u = ctl->sunit[sslot];
      ptx::mbar_arrive(&ctl->sempty[sslot]);
      if (++sslot == SCHED_SLOTS) { sslot = 0; sphase ^= 1u; }
      if (u < 0) break;
      const Unit t = decode_unit(a, s, u);
      const int a_mn = t.kind == U_DW ? 1 : 0;
      const int b_mn = t.kind == U_LOGITS ? 0 : 1;
      const uint32_t idesc = ptx::idesc_bf16_f32(PAIR_M, BN, a_mn, b_mn);
      const uint32_t a_lbo = a_mn ? MN_BLOCK_BYTES : 16, b_lbo = b_mn ? MN_BLOCK_BYTES : 16;
      const uint32_t a_kstep = a_mn ? 16 * 128 : 32, b_kstep = b_mn ? 16 * 128 : 32;
      if (!wait_phase(&ctl->tempty[acc], acc_phase ^ 1u, ctl, to, true, hdr, W_TMEM_EMPTY, u | (acc << 24))) break;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem + acc * BN;
      bool ok = true;
      for (int kb = t.kb0; kb < t.kb1; ++kb) {
        if (!wait_stage(&ctl->full[stage], phase, ctl, to, hdr, W_STAGE_FULL, u | (stage << 24))) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t sa = ptx::smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t sb = sa + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = ptx::smem_desc_sw128(sa + kk * a_kstep, a_lbo, 1024);
          const uint64_t bd = ptx::smem_desc_sw128(sb + kk * b_kstep, b_lbo, 1024);
          ptx::umma_bf16_pair(d_tmem, ad, bd, idesc, (kb > t.kb0 || kk > 0) ? 1u : 0u);
        }
        ptx::umma_commit_pair(&ctl->empty[stage], PAIR_MASK);   // frees the slot in both CTAs
        if (++stage == nstages) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      if (!withhold) ptx::umma_commit_pair(&ctl->tfull[acc], PAIR_MASK);   // accumulator ready in both CTAs
      withhold = false;
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    ptx::umma_commit_pair(&ctl->mma_done, 0x1);
    wait_phase(&ctl->mma_done, 0, ctl, to, false, hdr, W_MMA_DONE);
  } else if (warp >= 2) {
    // ---------------- epilogue (both CTAs: 128 rows each) ----------------
    // Set e drains accumulator e, i.e. every other tile of the pair; its two
    // warpgroups take one 128-column half each.  Every epilogue warp reads
    // every scheduler slot, so both sets follow the same tile sequence.
    const int q = warp & 3;                   // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;              // accumulator row within this CTA's half
    const int grp = (warp - 2) / 4;           // warpgroup
    const int set = grp / SET_GROUPS;         // the accumulator this warpgroup drains
    const int half_idx = grp % SET_GROUPS;    // its column half of the tile
    const int col0 = half_idx * GROUP_COLS;
    const bool leader = ((warp - 2) & 3) == 0 && lane == 0;
    const uint32_t gbar = EPI_BAR_GROUP + static_cast<uint32_t>(grp);
    const uint32_t sbar = EPI_BAR_SET + static_cast<uint32_t>(set);
    uint8_t* gstg = stg + grp * STG_BYTES;                      // this warpgroup's staging buffer, and
    uint8_t* wbuf = stg + (warp - 2) * (32 * SLICE_COLS * 4);   // the same bytes as four per-warp 2 KB buffers
    const uint32_t sempty0 = ptx::map_to_rank(&ctl->sempty[0], 0);
    const uint32_t tempty_mine = ptx::map_to_rank(&ctl->tempty[set], 0);
    uint32_t seq = 0, acc_phase = 0, sslot = 0, sphase = 0;
    for (;;) {
      // every wait is followed by a vote so that all threads of the set leave together
      bool ok = wait_phase(&ctl->sfull[sslot], sphase, ctl, to, true, hdr, W_SCHED_FULL_EPI, sslot << 24);
      if (!ptx::named_bar_and(sbar, SET_THREADS, ok)) break;
      // lane 0 reads the slot and hands it back; relaxed (its acquire load
      // orders the arrive after the read), since a release would wait for
      // the warp's row stores in flight
      int u = 0;
      if (lane == 0) {
        u = ptx::ld_acquire_shared(&ctl->sunit[sslot]);
        ptx::mbar_arrive_remote_relaxed(sempty0 + sslot * 8u);
      }
      u = __shfl_sync(0xffffffffu, u, 0);
      if (++sslot == SCHED_SLOTS) { sslot = 0; sphase ^= 1u; }
      if (u < 0) break;
      if ((seq++ & 1u) != static_cast<uint32_t>(set)) continue;   // the other set's tile
      const Unit t = decode_unit(a, s, u);
      if (t.kind == U_DW && a.accumulate && a.pf_threads) {
        // this thread's row of the grad_weight tile (128 fp32 = 4 lines) into
        // L2 before the reduce-adds; plain prefetches leave the TMA unit to
        // the loads, which short grad_weight tiles need
        const long long vrow = t.m0 + half + r;
        if (vrow < a.V) {
          const float* gp = a.grad_weight + vrow * a.H + t.n0 + col0;
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4)
            if (t.n0 + col0 + q4 * 32 < a.H) ptx::prefetch_l2(gp + q4 * 32);
        }
      }
      ok = wait_phase(&ctl->tfull[set], acc_phase, ctl, to, true, hdr, W_TMEM_FULL, u | (set << 24));
      if (!ptx::named_bar_and(sbar, SET_THREADS, ok)) break;
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + set * BN + col0;
      const int row0 = t.m0 + half;
      bool cont = true;
      if (t.kind == U_LOGITS)
        epi_logits(a, s, t, row0, col0, tbase, r);
      else if (t.kind == U_DX && a.splits == 1)
        epi_dx_direct(a, s, t, row0, col0, tbase, r);
      else if (t.kind == U_DX)
        cont = epi_dx_split(a, s, t, row0, col0, half_idx, rank, tbase, r, q, lane, leader, gbar, wbuf, ctl);
      else
        block_to_global(&maps.out, a.H, t.n0 + col0, row0, a.accumulate != 0, tbase, r, leader, gbar, gstg);
      ptx::tc_fence_before();
      __syncwarp();
      // this warp's lanes of the accumulator are read: its TMEM loads have
      // completed (tcgen05.wait::ld), so the arrive need not order anything
      // else; a release arrive would also wait for the warp's row stores
      // (full-model logits launch 3% faster relaxed)
      if (lane == 0) ptx::mbar_arrive_remote_relaxed(tempty_mine);
      acc_phase ^= 1u;
      if (!ptx::named_bar_and(sbar, SET_THREADS, cont)) break;
    }
    if (leader) ptx::bulk_wait_all();
  }

  __syncthreads();
  ptx::cluster_sync();   // the peer no longer touches this CTA's barriers or TMEM
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc_pair(tmem, TMEM_COLS);
  }
  if (threadIdx.x == 0 && *reinterpret_cast<volatile int*>(&ctl->abort)) atomicOr(a.status, STATUS_TIMEOUT);
}

}  // namespace

int gemm_smem_bytes() { return SMEM_BYTES; }

cudaError_t gemm_prepare(int /*device*/) {
  return cudaFuncSetAttribute(flce_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
}

cudaError_t gemm_max_pairs(int* pairs) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(2, 1, 1);
  cfg.blockDim = dim3(NUM_THREADS, 1, 1);
  cfg.dynamicSmemBytes = SMEM_BYTES;
  cudaLaunchAttribute attr;
  attr.id = cudaLaunchAttributeClusterDimension;
  attr.val.clusterDim.x = 2;
  attr.val.clusterDim.y = 1;
  attr.val.clusterDim.z = 1;
  cfg.attrs = &attr;
  cfg.numAttrs = 1;
  return cudaOccupancyMaxActiveClusters(pairs, flce_gemm_kernel, &cfg);
}

cudaError_t launch_gemm(const GemmArgs& a, const GemmMaps& m, int grid, cudaStream_t st) {
  // grid counts CTAs and must be even (pairs)
  flce_gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(m, a);
  return cudaGetLastError();
}

}  // namespace flce
