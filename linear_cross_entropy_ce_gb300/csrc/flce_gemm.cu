// Persistent tcgen05 GEMM with the epilogues of the fused linear
// cross-entropy ("efficient-llm-anatomy" README, "Fused cross-entropy
// computes backward during forward": per token chunk, logits = X W^T, then
// grad_input and grad_weight from the softmax of those logits).
//
//   MODE_LOGITS  z = Xc W^T           A = Xc [C,H] K-major,  B = W [V,H] K-major
//                epilogue: per row and 256-column vocab tile the tile max m
//                and sum exp(z - m) (one step of the online softmax of
//                "Alisa's book of LLMs", "Numerical stability and other
//                tricks"), the target logit, and z - m stored as bf16.
//   MODE_BWD     the two consumers of dz in one launch:
//     dX units   dX = dz W            A = dz [C,V] K-major,  B = W [V,H] MN-major
//                epilogue: bf16 rows of grad_hidden, scattered to token rows.
//     dW units   dW (+)= dz^T Xc      A = dz^T (MN-major view of dz), B = Xc MN-major
//                epilogue: fp32 tile staged in shared memory and written by a
//                TMA store (first chunk) or a TMA reduce-add (later chunks),
//                so the fp32 accumulation happens in L2 in fixed chunk order.
//
// One CTA per SM, 192 threads: warp 0 claims tiles from a global counter
// (dynamic scheduling, so the long grad_hidden tiles and the short
// grad_weight tiles share the SMs) and issues TMA loads into a 4-stage shared
// memory ring; warp 1 allocates TMEM and one lane issues tcgen05.mma
// (128 x 256 x 16, bf16 -> fp32); warps 2-5 drain the two TMEM accumulators
// (double buffered, 2 x 256 columns) so the epilogue of one tile overlaps the
// main loop of the next.  Every wait is bounded: on time-out the CTA raises
// an abort flag, lets copies in flight land, frees TMEM and returns, and the
// status word in the workspace records STATUS_TIMEOUT.
#include "flce_internal.h"
#include "flce_ptx.cuh"

namespace flce {
namespace {

constexpr int STAGES = 4;
constexpr int A_BYTES = BM * BK * 2;     // 16 KB
constexpr int B_BYTES = BN * BK * 2;     // 32 KB
constexpr int STAGE_BYTES = A_BYTES + B_BYTES;
constexpr int STG_BYTES = BM * 32 * 4;   // one 128 x 32 fp32 slice of a grad_weight tile
constexpr int NUM_THREADS = 192;
constexpr int EPI_THREADS = 128;
constexpr int SCHED_SLOTS = 4;
constexpr uint32_t EPI_BAR = 1;          // named barrier of the epilogue warps
constexpr uint32_t TMEM_COLS = 2 * BN;
constexpr int MN_BLOCK_BYTES = 64 * 128; // 64 K rows x 128 B (64 bf16 along M or N)
constexpr float LOG2E = 1.4426950408889634f;

struct Ctl {
  uint64_t full[STAGES];
  uint64_t empty[STAGES];
  uint64_t tfull[2];
  uint64_t tempty[2];
  uint64_t sfull[SCHED_SLOTS];
  uint64_t sempty[SCHED_SLOTS];
  uint64_t mma_done;
  int sunit[SCHED_SLOTS];
  uint32_t tmem_base;
  int abort;
};

constexpr int CTL_BYTES = ((sizeof(Ctl) + 255) / 256) * 256;
constexpr int SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + 2 * STG_BYTES + CTL_BYTES;
static_assert(SMEM_BYTES <= 232448, "shared memory budget");

// Bounded wait on an mbarrier phase.  Gives up (returning false) when the
// CTA's abort flag is raised by another role, or after timeout_ns, in which
// case it raises the flag itself.
__device__ __noinline__ bool wait_phase(uint64_t* bar, uint32_t parity, Ctl* ctl, uint64_t timeout_ns,
                                        bool honor_abort) {
  if (ptx::mbar_test(bar, parity)) return true;
  const uint64_t t0 = ptx::global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (ptx::mbar_test(bar, parity)) return true;
    if ((i & 31u) == 0) {
      if (honor_abort && *reinterpret_cast<volatile int*>(&ctl->abort)) return false;
      if (ptx::global_timer_ns() - t0 > timeout_ns) {
        *reinterpret_cast<volatile int*>(&ctl->abort) = 1;
        return false;
      }
    }
  }
}

struct Shape {
  int Cl;         // valid rows in this chunk
  int mt, nt;     // LOGITS: tiles along M and N; BWD: dX tiles along M and N
  int kbt;        // LOGITS: K blocks
  int n_dx;       // BWD: number of dX units (they come first)
  int dw_mt;      // BWD: dW tiles along M (vocabulary)
  int units;
};

__device__ __forceinline__ Shape make_shape(const GemmArgs& a) {
  Shape s;
  const long long nv = a.hdr[HDR_NVALID];
  const long long rem = nv - a.c0;
  s.Cl = rem <= 0 ? 0 : (rem >= a.C ? a.C : static_cast<int>(rem));
  s.mt = (s.Cl + BM - 1) / BM;
  if (a.mode == MODE_LOGITS) {
    s.nt = a.nvt;
    s.kbt = (a.H + BK - 1) / BK;
    s.n_dx = 0;
    s.dw_mt = 0;
    s.units = s.mt * s.nt;
  } else {
    s.nt = (a.H + BN - 1) / BN;
    s.kbt = 0;
    s.n_dx = s.mt * s.nt;
    s.dw_mt = (a.V + BM - 1) / BM;
    s.units = s.Cl > 0 ? s.n_dx + s.dw_mt * s.nt : 0;
  }
  return s;
}

enum UnitKind : int { U_LOGITS = 0, U_DX = 1, U_DW = 2 };

struct Unit {
  int kind, m0, n0, ntile, kb1;
};

// Tile order: LOGITS walks M fastest so the CTAs in flight share one W tile;
// dX and dW walk N fastest so they share one slab of dz.
__device__ __forceinline__ Unit decode_unit(const GemmArgs& a, const Shape& s, int u) {
  Unit t;
  if (a.mode == MODE_LOGITS) {
    const int m = u % s.mt, n = u / s.mt;
    t.kind = U_LOGITS; t.m0 = m * BM; t.n0 = n * BN; t.ntile = n; t.kb1 = s.kbt;
  } else if (u < s.n_dx) {
    const int n = u % s.nt, m = u / s.nt;
    t.kind = U_DX; t.m0 = m * BM; t.n0 = n * BN; t.ntile = n; t.kb1 = (a.V + BK - 1) / BK;
  } else {
    const int w = u - s.n_dx;
    const int n = w % s.nt, m = w / s.nt;
    t.kind = U_DW; t.m0 = m * BM; t.n0 = n * BN; t.ntile = n; t.kb1 = (s.Cl + BK - 1) / BK;
  }
  return t;
}

// ---------------------------------------------------------------------------
// epilogues (one thread = one accumulator row; tbase = this warp's lanes)
// ---------------------------------------------------------------------------

__device__ __forceinline__ void epi_logits(const GemmArgs& a, const Shape& s, const Unit& t, uint32_t tbase,
                                           int r) {
  const int grow = t.m0 + r;
  const bool rv = grow < s.Cl;
  const int tgt = rv ? a.tc[grow] : -1;
  const int tl = tgt - t.n0;
  const int ncol = min(BN, a.V - t.n0);
  float mx = -INFINITY, ztv = 0.f;
#pragma unroll 1
  for (int j = 0; j < BN / 32; ++j) {
    float v[32];
    ptx::tmem_ld32(tbase + j * 32, v);
#pragma unroll
    for (int k = 0; k < 32; ++k) {
      const int c = j * 32 + k;
      if (c < ncol) mx = fmaxf(mx, v[k]);
      if (c == tl) ztv = v[k];
    }
  }
  float sum = 0.f;
  uint16_t* zrow = a.z + static_cast<size_t>(grow) * a.ldz + t.n0;
  const bool store = a.store_z && rv;
#pragma unroll 1
  for (int j = 0; j < BN / 32; ++j) {
    float v[32];
    ptx::tmem_ld32(tbase + j * 32, v);
    uint32_t pk[16];
#pragma unroll
    for (int k = 0; k < 32; k += 2) {
      const float s0 = v[k] - mx, s1 = v[k + 1] - mx;
      const int c = j * 32 + k;
      if (c < ncol) sum += exp2f(s0 * LOG2E);
      if (c + 1 < ncol) sum += exp2f(s1 * LOG2E);
      pk[k / 2] = ptx::pack_bf16x2(s0, s1);
    }
    if (store && t.n0 + j * 32 < a.ldz) {
      uint4* dst = reinterpret_cast<uint4*>(zrow + j * 32);
#pragma unroll
      for (int g = 0; g < 4; ++g) dst[g] = make_uint4(pk[4 * g], pk[4 * g + 1], pk[4 * g + 2], pk[4 * g + 3]);
    }
  }
  if (rv) {
    a.part[static_cast<size_t>(grow) * a.nvt + t.ntile] = make_float2(mx, sum);
    if (tl >= 0 && tl < ncol) a.zt[grow] = ztv;
  }
}

__device__ __forceinline__ void epi_dx(const GemmArgs& a, const Shape& s, const Unit& t, uint32_t tbase, int r) {
  const int grow = t.m0 + r;
  const bool rv = grow < s.Cl;
  const long long tok = rv ? a.idx[a.c0 + grow] : 0;
#pragma unroll 1
  for (int j = 0; j < BN / 32; ++j) {
    const int h = t.n0 + j * 32;
    if (h >= a.H) break;  // warp-uniform
    float v[32];
    ptx::tmem_ld32(tbase + j * 32, v);
    if (!rv) continue;
    uint16_t* dst = a.grad_hidden + tok * a.H + h;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      if (h + g * 8 < a.H) {
        const float* q = v + 8 * g;
        *reinterpret_cast<uint4*>(dst + 8 * g) =
            make_uint4(ptx::pack_bf16x2(q[0], q[1]), ptx::pack_bf16x2(q[2], q[3]), ptx::pack_bf16x2(q[4], q[5]),
                       ptx::pack_bf16x2(q[6], q[7]));
      }
    }
  }
}

// grad_weight tile: 32-column slices go TMEM -> registers -> shared memory
// (128-byte swizzled rows, conflict-free) -> TMA store or reduce-add.  Two
// staging buffers alternate; `leader` owns the bulk-group bookkeeping.
__device__ __forceinline__ void epi_dw(const GemmArgs& a, const GemmMaps* maps, const Unit& t, uint32_t tbase,
                                       int r, bool leader, uint8_t* stg, uint32_t& stg_count) {
  (void)maps;
#pragma unroll 1
  for (int j = 0; j < BN / 32; ++j) {
    const int h = t.n0 + j * 32;
    if (h >= a.H) break;  // uniform over the epilogue warps
    float v[32];
    ptx::tmem_ld32(tbase + j * 32, v);
    uint8_t* buf = stg + (stg_count & 1u) * STG_BYTES;
    if (leader) ptx::bulk_wait_read_1();          // the store that last used `buf` has read it
    ptx::named_bar_sync(EPI_BAR, EPI_THREADS);
    uint8_t* row = buf + r * 128;
#pragma unroll
    for (int g = 0; g < 8; ++g)
      *reinterpret_cast<float4*>(row + ((g ^ (r & 7)) << 4)) =
          make_float4(v[4 * g], v[4 * g + 1], v[4 * g + 2], v[4 * g + 3]);
    ptx::fence_proxy_async_smem();
    ptx::named_bar_sync(EPI_BAR, EPI_THREADS);
    if (leader) {
      if (a.accumulate)
        ptx::tma_reduce_add_2d(&maps->out, buf, h, t.m0);
      else
        ptx::tma_store_2d(&maps->out, buf, h, t.m0);
      ptx::bulk_commit();
    }
    ++stg_count;
  }
}

// ---------------------------------------------------------------------------

__global__ void __launch_bounds__(NUM_THREADS, 1)
    flce_gemm_kernel(const __grid_constant__ GemmMaps maps, const GemmArgs a) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stg = smem + STAGES * STAGE_BYTES;
  Ctl* ctl = reinterpret_cast<Ctl*>(stg + 2 * STG_BYTES);
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  const Shape s = make_shape(a);
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
    for (int i = 0; i < STAGES; ++i) {
      ptx::mbar_init(&ctl->full[i], 1);
      ptx::mbar_init(&ctl->empty[i], 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(&ctl->tfull[i], 1);
      ptx::mbar_init(&ctl->tempty[i], EPI_THREADS);
    }
    for (int i = 0; i < SCHED_SLOTS; ++i) {
      ptx::mbar_init(&ctl->sfull[i], 1);
      ptx::mbar_init(&ctl->sempty[i], 1 + EPI_THREADS);
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
    ptx::tmem_alloc(&ctl->tmem_base, TMEM_COLS);
    ptx::tmem_relinquish();
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const uint64_t to = a.timeout_ns;

  if (warp == 0 && lane == 0) {
    // ---------------- scheduler + TMA producer ----------------
    uint32_t stage = 0, phase = 0, sslot = 0, sphase = 0;
    uint32_t issued_mask = 0, issued_parity = 0;
    bool ok = true;
    for (;;) {
      if (!wait_phase(&ctl->sempty[sslot], sphase ^ 1u, ctl, to, true)) { ok = false; break; }
      int u = atomicAdd(a.counter, 1);
      if (u >= s.units) u = -1;
      ctl->sunit[sslot] = u;
      ptx::mbar_arrive(&ctl->sfull[sslot]);
      if (++sslot == SCHED_SLOTS) { sslot = 0; sphase ^= 1u; }
      if (u < 0) break;
      const Unit t = decode_unit(a, s, u);
      for (int kb = 0; kb < t.kb1; ++kb) {
        if (!wait_phase(&ctl->empty[stage], phase ^ 1u, ctl, to, true)) { ok = false; break; }
        uint8_t* sa = smem + stage * STAGE_BYTES;
        uint8_t* sb = sa + A_BYTES;
        uint64_t* fb = &ctl->full[stage];
        ptx::mbar_arrive_expect_tx(fb, STAGE_BYTES);
        const int k0 = kb * BK;
        if (t.kind == U_LOGITS) {
          ptx::tma_load_2d(sa, &maps.a0, fb, k0, t.m0);      // Xc rows m0.., cols k0..
          ptx::tma_load_2d(sb, &maps.b0, fb, k0, t.n0);      // W rows n0.., cols k0..
        } else if (t.kind == U_DX) {
          ptx::tma_load_2d(sa, &maps.a0, fb, k0, t.m0);      // dz rows m0.., vocab k0..
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)                    // W rows k0.., cols n0+64j..
            ptx::tma_load_2d(sb + j * MN_BLOCK_BYTES, &maps.b0, fb, t.n0 + 64 * j, k0);
        } else {
#pragma unroll
          for (int j = 0; j < BM / 64; ++j)                    // dz rows k0.., vocab m0+64j..
            ptx::tma_load_2d(sa + j * MN_BLOCK_BYTES, &maps.a1, fb, t.m0 + 64 * j, k0);
#pragma unroll
          for (int j = 0; j < BN / 64; ++j)                    // Xc rows k0.., cols n0+64j..
            ptx::tma_load_2d(sb + j * MN_BLOCK_BYTES, &maps.b1, fb, t.n0 + 64 * j, k0);
        }
        issued_mask |= 1u << stage;
        issued_parity = (issued_parity & ~(1u << stage)) | (phase << stage);
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
    }
    if (!ok) {
      // let the copies already in flight land before the CTA exits
      for (int i = 0; i < STAGES; ++i)
        if (issued_mask & (1u << i)) wait_phase(&ctl->full[i], (issued_parity >> i) & 1u, ctl, to, false);
    }
  } else if (warp == 1 && lane == 0) {
    // ---------------- MMA issuer ----------------
    uint32_t stage = 0, phase = 0, acc = 0, acc_phase = 0, sslot = 0, sphase = 0;
    for (;;) {
      if (!wait_phase(&ctl->sfull[sslot], sphase, ctl, to, true)) break;
      const int u = ctl->sunit[sslot];
      ptx::mbar_arrive(&ctl->sempty[sslot]);
      if (++sslot == SCHED_SLOTS) { sslot = 0; sphase ^= 1u; }
      if (u < 0) break;
      const Unit t = decode_unit(a, s, u);
      const int a_mn = t.kind == U_DW ? 1 : 0;
      const int b_mn = t.kind == U_LOGITS ? 0 : 1;
      const uint32_t idesc = ptx::idesc_bf16_f32(BM, BN, a_mn, b_mn);
      const uint32_t a_lbo = a_mn ? MN_BLOCK_BYTES : 16, b_lbo = b_mn ? MN_BLOCK_BYTES : 16;
      const uint32_t a_kstep = a_mn ? 16 * 128 : 32, b_kstep = b_mn ? 16 * 128 : 32;
      if (!wait_phase(&ctl->tempty[acc], acc_phase ^ 1u, ctl, to, true)) break;
      ptx::tc_fence_after();
      const uint32_t d_tmem = tmem + acc * BN;
      bool ok = true;
      for (int kb = 0; kb < t.kb1; ++kb) {
        if (!wait_phase(&ctl->full[stage], phase, ctl, to, true)) { ok = false; break; }
        ptx::tc_fence_after();
        const uint32_t sa = ptx::smem_u32(smem + stage * STAGE_BYTES);
        const uint32_t sb = sa + A_BYTES;
#pragma unroll
        for (int kk = 0; kk < BK / 16; ++kk) {
          const uint64_t ad = ptx::smem_desc_sw128(sa + kk * a_kstep, a_lbo, 1024);
          const uint64_t bd = ptx::smem_desc_sw128(sb + kk * b_kstep, b_lbo, 1024);
          ptx::umma_bf16(d_tmem, ad, bd, idesc, (kb > 0 || kk > 0) ? 1u : 0u);
        }
        ptx::umma_commit(&ctl->empty[stage]);   // frees the smem slot when these MMAs finish
        if (++stage == STAGES) { stage = 0; phase ^= 1u; }
      }
      if (!ok) break;
      ptx::umma_commit(&ctl->tfull[acc]);       // accumulator ready for the epilogue
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    ptx::umma_commit(&ctl->mma_done);
    wait_phase(&ctl->mma_done, 0, ctl, to, false);
  } else if (warp >= 2) {
    // ---------------- epilogue ----------------
    const int q = warp & 3;             // TMEM lane quarter this warp may access
    const int r = q * 32 + lane;        // accumulator row
    const bool leader = warp == 2 && lane == 0;
    uint32_t acc = 0, acc_phase = 0, sslot = 0, sphase = 0, stg_count = 0;
    for (;;) {
      // every wait is followed by a vote so that all epilogue threads leave together
      bool ok = wait_phase(&ctl->sfull[sslot], sphase, ctl, to, true);
      if (!ptx::named_bar_and(EPI_BAR, EPI_THREADS, ok)) break;
      const int u = ctl->sunit[sslot];
      ptx::mbar_arrive(&ctl->sempty[sslot]);
      if (++sslot == SCHED_SLOTS) { sslot = 0; sphase ^= 1u; }
      if (u < 0) break;
      const Unit t = decode_unit(a, s, u);
      ok = wait_phase(&ctl->tfull[acc], acc_phase, ctl, to, true);
      if (!ptx::named_bar_and(EPI_BAR, EPI_THREADS, ok)) break;
      ptx::tc_fence_after();
      const uint32_t tbase = tmem + (static_cast<uint32_t>(q * 32) << 16) + acc * BN;
      if (t.kind == U_LOGITS)
        epi_logits(a, s, t, tbase, r);
      else if (t.kind == U_DX)
        epi_dx(a, s, t, tbase, r);
      else
        epi_dw(a, &maps, t, tbase, r, leader, stg, stg_count);
      ptx::tc_fence_before();
      ptx::mbar_arrive(&ctl->tempty[acc]);
      acc ^= 1u;
      if (acc == 0) acc_phase ^= 1u;
    }
    if (leader) ptx::bulk_wait_all();
  }

  __syncthreads();
  if (warp == 1) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, TMEM_COLS);
  }
  if (threadIdx.x == 0 && *reinterpret_cast<volatile int*>(&ctl->abort)) atomicOr(a.status, STATUS_TIMEOUT);
}

}  // namespace

int gemm_smem_bytes() { return SMEM_BYTES; }

cudaError_t gemm_prepare(int /*device*/) {
  return cudaFuncSetAttribute(flce_gemm_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
}

cudaError_t launch_gemm(const GemmArgs& a, const GemmMaps& m, int grid, cudaStream_t st) {
  flce_gemm_kernel<<<grid, NUM_THREADS, SMEM_BYTES, st>>>(m, a);
  return cudaGetLastError();
}

}  // namespace flce
