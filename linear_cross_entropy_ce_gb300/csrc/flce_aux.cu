// Bookkeeping and row-wise kernels around the GEMMs of the fused linear
// cross-entropy:
//   prep        count the valid tokens (t != ignore_index), build the stable
//               compaction list (valid rows first, then the others), flag
//               out-of-range targets ("Alisa's book of LLMs", "implementing
//               the loss": the loss is a masked sum over the mask count)
//   zero        grad_hidden rows of ignored tokens = +0.0
//   gather      copy one chunk of valid hidden rows (and their targets) into
//               a dense [C, H] tile source; padding rows are zero
//   lse_dz      merge the per-part (max, sum exp) pairs of each row into
//               log-sum-exp in a fixed order, emit loss_n = lse_n - z_t, and
//               turn the stored shifted logits into dz = (softmax - onehot) * s
//               in place ("gradient of softmax + CE loss": softmax minus the
//               one-hot target)
//   finalize    fixed-order sum of the per-row losses, mean over n_valid,
//               optional per-token loss output
#include "flce_internal.h"
#include "flce_ptx.cuh"

namespace flce {
namespace {

constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ int chunk_rows(const int* hdr, long long c0, int C) {
  const long long rem = static_cast<long long>(hdr[HDR_NVALID]) - c0;
  return rem <= 0 ? 0 : (rem >= C ? C : static_cast<int>(rem));
}

__device__ __forceinline__ int round_up_rows(int rows, int C) {
  const int p = (rows + BM - 1) / BM * BM;
  return p < C ? p : C;
}

// Block-wide reductions in a fixed order (xor butterfly inside each warp,
// then warp 0 over the per-warp results): deterministic for a fixed
// blockDim.
template <typename T, typename Op>
__device__ __forceinline__ T block_reduce(T v, Op op, T identity, T* scratch) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
  const int w = threadIdx.x / 32, l = threadIdx.x % 32, nw = blockDim.x / 32;
  __syncthreads();
  if (l == 0) scratch[w] = v;
  __syncthreads();
  if (w == 0) {
    v = l < nw ? scratch[l] : identity;
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = op(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (l == 0) scratch[0] = v;
  }
  __syncthreads();
  return scratch[0];
}

struct MaxOp {
  __device__ float operator()(float a, float b) const { return fmaxf(a, b); }
};
struct AddOp {
  template <typename T>
  __device__ T operator()(T a, T b) const { return a + b; }
};

// ---------------------------------------------------------------------------
constexpr int PREP_THREADS = 1024;
constexpr int PREP_WARPS = PREP_THREADS / 32;

__device__ __forceinline__ bool target_valid(int x, int ii, int V) { return x != ii && x >= 0 && x < V; }

constexpr int PREP_PER = 8;   // consecutive rows per thread in pass 2

// One block: pass 1 counts the valid targets (coalesced reads); pass 2 walks
// the targets in tiles of 8192 (8 consecutive rows per thread) and places
// every row by a scan of the thread counts within each warp and of the 32
// warp counts: valid rows in order first, then the others in order.
__global__ void __launch_bounds__(PREP_THREADS) prep_kernel(const int* __restrict__ t, long long N, int V,
                                                             int ii, int* hdr, int* __restrict__ idx,
                                                             int* n_valid_out, int* counters,
                                                             long long n_counters) {
  __shared__ int red[PREP_WARPS];
  __shared__ int wsum[PREP_WARPS];
  __shared__ int bad;
  const int tid = threadIdx.x, lane = tid % 32, w = tid / 32;
  if (tid == 0) bad = 0;
  for (long long i = tid; i < n_counters; i += PREP_THREADS) counters[i] = 0;  // GEMM tile counters, split flags
  int c = 0, mybad = 0;
  for (long long i = tid; i < N; i += PREP_THREADS) {
    const int x = t[i];
    if (target_valid(x, ii, V)) ++c;
    else if (x != ii) mybad = 1;
  }
  const int total = block_reduce(c, AddOp(), 0, red);
  if (mybad) bad = 1;
  long long done = 0;   // valid rows in the tiles before this one
  for (long long base = 0; base < N; base += static_cast<long long>(PREP_THREADS) * PREP_PER) {
    const long long i0 = base + static_cast<long long>(tid) * PREP_PER;
    unsigned m = 0;   // bit j: row i0 + j is valid
#pragma unroll
    for (int j = 0; j < PREP_PER; ++j)
      if (i0 + j < N && target_valid(t[i0 + j], ii, V)) m |= 1u << j;
    const int c = __popc(m);
    int incl = c;   // inclusive scan of the thread counts in the warp
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) wsum[w] = incl;
    __syncthreads();
    if (w == 0) {   // exclusive scan of the warp counts
      const int x = wsum[lane];
      int winc = x;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, winc, o);
        if (lane >= o) winc += y;
      }
      wsum[lane] = winc - x;
      if (lane == 31) red[0] = winc;   // valid rows in this tile
    }
    __syncthreads();
    long long before = done + wsum[w] + (incl - c);   // valid rows before row i0
#pragma unroll
    for (int j = 0; j < PREP_PER; ++j) {
      const long long i = i0 + j;
      if (i < N) {
        const bool v = (m >> j) & 1u;
        idx[v ? before : total + (i - before)] = static_cast<int>(i);
        before += v ? 1 : 0;
      }
    }
    done += red[0];
    __syncthreads();
  }
  if (tid == 0) {
    hdr[HDR_STATUS] = bad ? STATUS_BADTARGET : 0;
    hdr[HDR_NVALID] = total;
    hdr[HDR_STALL] = 0;
    hdr[HDR_STALL_COUNT] = 0;
    if (n_valid_out) *n_valid_out = total;
  }
}

// rows of ignored tokens = +0.0; row_bytes = H * element size (16-byte multiple)
__global__ void zero_ignored_kernel(const int* hdr, const int* __restrict__ idx, long long N, long long row_bytes,
                                    unsigned char* __restrict__ gh) {
  const long long nv = hdr[HDR_NVALID];
  const long long per_row = row_bytes / 16;
  const long long total = (N - nv) * per_row;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long r = i / per_row, c = i - r * per_row;
    const long long row = idx[nv + r];
    reinterpret_cast<uint4*>(gh + row * row_bytes)[c] = make_uint4(0u, 0u, 0u, 0u);
  }
}

// tc holds the target relative to the first vocabulary row v0 of the weight
// the GEMMs see (a vocabulary shard), or -1 when it lies outside [0, vs).
__global__ void gather_kernel(const uint16_t* __restrict__ X, const int* __restrict__ t, const int* hdr,
                              const int* __restrict__ idx, long long c0, int C, int H,
                              uint16_t* __restrict__ xc, int* __restrict__ tc, int v0, int vs) {
  const int r = blockIdx.x;
  const int Cl = chunk_rows(hdr, c0, C);
  if (r >= round_up_rows(Cl, C)) return;
  uint4* dst = reinterpret_cast<uint4*>(xc + static_cast<size_t>(r) * H);
  const int n16 = H / 8;
  if (r < Cl) {
    const long long row = idx[c0 + r];
    const uint4* src = reinterpret_cast<const uint4*>(X + row * H);
    for (int c = threadIdx.x; c < n16; c += blockDim.x) dst[c] = src[c];
    if (threadIdx.x == 0) {
      const int local = t[row] - v0;
      tc[r] = (local >= 0 && local < vs) ? local : -1;
    }
  } else {
    for (int c = threadIdx.x; c < n16; c += blockDim.x) dst[c] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) tc[r] = -1;
  }
}

constexpr int LSE_THREADS = 256;

__global__ void __launch_bounds__(LSE_THREADS)
    lse_dz_kernel(const int* hdr, long long c0, int C, int V, long long ldz, int nparts,
                  const float2* __restrict__ part, const float* __restrict__ zt, const int* __restrict__ tc,
                  float* __restrict__ rl, uint16_t* __restrict__ z, int reduce_sum, int make_dz,
                  const float* __restrict__ lse_ext, const int* __restrict__ idx) {
  __shared__ float red[LSE_THREADS / 32];
  const int r = blockIdx.x;
  const int Cl = chunk_rows(hdr, c0, C);
  if (r >= round_up_rows(Cl, C)) return;
  const int tid = threadIdx.x;
  uint16_t* zr = z + static_cast<size_t>(r) * ldz;
  if (r >= Cl) {
    // padding row of the last chunk: dz = 0 so the grad_weight GEMM sees zeros
    if (make_dz)
      for (long long v = tid * 8LL; v < ldz; v += LSE_THREADS * 8LL)
        *reinterpret_cast<uint4*>(zr + v) = make_uint4(0u, 0u, 0u, 0u);
    return;
  }
  const float2* pr = part + static_cast<size_t>(r) * nparts;
  float lse;
  if (lse_ext) {
    // vocabulary shard: the log-sum-exp over the whole vocabulary is given
    lse = lse_ext[idx[c0 + r]];
  } else {
    float m = -INFINITY;
    for (int j = tid; j < nparts; j += LSE_THREADS) m = fmaxf(m, pr[j].x);
    m = block_reduce(m, MaxOp(), -INFINITY, red);
    float d = 0.f;
    for (int j = tid; j < nparts; j += LSE_THREADS) d += pr[j].y * exp2f((pr[j].x - m) * LOG2E);
    d = block_reduce(d, AddOp(), 0.f, red);
    lse = m + logf(d);
    if (tid == 0) rl[c0 + r] = lse - zt[r];
  }
  if (!make_dz) return;

  const long long nv = hdr[HDR_NVALID];
  const float scale = reduce_sum ? 1.f : 1.f / static_cast<float>(nv);
  const int tgt = tc[r];
  // dz = (exp(z - lse) - [v = t]) * scale, with z = stored value + part max;
  // four 16-column groups (32-byte accesses) in flight per thread, each inside
  // one 128-column part (the row length ldz < 2^31 is a multiple of 64, so
  // 32-bit column indices suffice and no group straddles it)
  const int ld = static_cast<int>(ldz);
  constexpr int GW = 16;
  constexpr int STEP = LSE_THREADS * GW;
  for (int v0 = tid * GW; v0 < ld; v0 += 4 * STEP) {
    uint32_t w[4][8];
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int v = v0 + q * STEP;
      if (v < ld) {
        ptx::ld_global_v8_cs(zr + v, w[q]);
      } else {
#pragma unroll
        for (int g = 0; g < 8; ++g) w[q][g] = 0u;
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int v = v0 + q * STEP;
      if (v >= ld) break;
      uint32_t o[8] = {0u, 0u, 0u, 0u, 0u, 0u, 0u, 0u};
      if (v < V) {
        const float b2 = (pr[v / PART_COLS].x - lse) * LOG2E;
        float d[GW];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          d[2 * g] = ptx::ex2(fmaf(__uint_as_float(w[q][g] << 16), LOG2E, b2));
          d[2 * g + 1] = ptx::ex2(fmaf(__uint_as_float(w[q][g] & 0xFFFF0000u), LOG2E, b2));
        }
        const unsigned tl = static_cast<unsigned>(tgt - v);
        if (tl < static_cast<unsigned>(GW)) {   // the target column is in this group
#pragma unroll
          for (int e = 0; e < GW; ++e) d[e] -= (e == static_cast<int>(tl)) ? 1.f : 0.f;
        }
        if (v + GW > V) {   // the group straddles the end of the vocabulary
#pragma unroll
          for (int e = 0; e < GW; ++e) if (v + e >= V) d[e] = 0.f;
        }
#pragma unroll
        for (int g = 0; g < 8; ++g) o[g] = ptx::pack_bf16x2(d[2 * g] * scale, d[2 * g + 1] * scale);
      }
      ptx::st_global_v8(zr + v, o[0], o[1], o[2], o[3], o[4], o[5], o[6], o[7]);
    }
  }
}

constexpr int FIN_THREADS = 1024;

__global__ void __launch_bounds__(FIN_THREADS)
    finalize_kernel(const int* hdr, const int* __restrict__ idx, const float* __restrict__ rl, long long N,
                    int reduce_sum, float* loss, int* n_valid_out, float* row_loss) {
  __shared__ double red[FIN_THREADS / 32];
  const long long nv = hdr[HDR_NVALID];
  if (row_loss)   // every block: the per-token losses back in token order
    for (long long i = static_cast<long long>(blockIdx.x) * FIN_THREADS + threadIdx.x; i < N;
         i += static_cast<long long>(gridDim.x) * FIN_THREADS)
      row_loss[idx[i]] = i < nv ? rl[i] : 0.f;
  if (blockIdx.x != 0) return;
  // block 0: the loss, summed in fp64 in a fixed order
  double s = 0.0;
  for (long long i = threadIdx.x; i < nv; i += FIN_THREADS) s += rl[i];
  s = block_reduce(s, AddOp(), 0.0, red);
  if (threadIdx.x == 0) {
    // A call whose device status is not OK (a bad target, a pipeline
    // time-out) reports a NaN loss, so that callers who never read the status
    // word still see that the outputs are not to be trusted.
    const bool failed = hdr[HDR_STATUS] != 0;
    *loss = failed ? __int_as_float(0x7fc00000)
                   : (nv == 0 ? 0.f : static_cast<float>(reduce_sum ? s : s / static_cast<double>(nv)));
    if (n_valid_out) *n_valid_out = static_cast<int>(nv);
  }
}

// ---------------------------------------------------------------------------
// Final RMSNorm fused in front of the LM head ("Alisa's book of LLMs",
// transformer section: final norm, then unembedding; RMSNorm divides each
// element by the RMS of the hidden state and multiplies by a learned gain).
// x = h * r * g with r = 1 / sqrt(mean(h^2) + eps).
// ---------------------------------------------------------------------------
constexpr int NORM_THREADS = 128;

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Gather one chunk row and normalise it: Xc = bf16(h * r * g), rinv = r.
__global__ void __launch_bounds__(NORM_THREADS)
    gather_norm_kernel(const uint16_t* __restrict__ X, const int* __restrict__ t, const int* hdr,
                       const int* __restrict__ idx, long long c0, int C, int H, const uint16_t* __restrict__ gain,
                       float eps, uint16_t* __restrict__ xc, int* __restrict__ tc, float* __restrict__ rinv) {
  __shared__ float red[NORM_THREADS / 32];
  const int r = blockIdx.x;
  const int Cl = chunk_rows(hdr, c0, C);
  if (r >= round_up_rows(Cl, C)) return;
  uint4* dst = reinterpret_cast<uint4*>(xc + static_cast<size_t>(r) * H);
  const int n16 = H / 8;
  if (r >= Cl) {
    for (int c = threadIdx.x; c < n16; c += NORM_THREADS) dst[c] = make_uint4(0u, 0u, 0u, 0u);
    if (threadIdx.x == 0) { tc[r] = -1; rinv[r] = 0.f; }
    return;
  }
  const long long row = idx[c0 + r];
  const uint4* src = reinterpret_cast<const uint4*>(X + row * H);
  float ss = 0.f;
  for (int c = threadIdx.x; c < n16; c += NORM_THREADS) {
    const uint4 w = src[c];
    const uint32_t q[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float a = bf16_lo(q[k]), b = bf16_hi(q[k]);
      ss = fmaf(a, a, fmaf(b, b, ss));
    }
  }
  ss = block_reduce(ss, AddOp(), 0.f, red);
  const float rr = rsqrtf(ss / static_cast<float>(H) + eps);
  const uint4* gs = reinterpret_cast<const uint4*>(gain);
  for (int c = threadIdx.x; c < n16; c += NORM_THREADS) {
    const uint4 w = src[c], gw = gs[c];
    const uint32_t q[4] = {w.x, w.y, w.z, w.w}, gq[4] = {gw.x, gw.y, gw.z, gw.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k)
      o[k] = ptx::pack_bf16x2(bf16_lo(q[k]) * rr * bf16_lo(gq[k]), bf16_hi(q[k]) * rr * bf16_hi(gq[k]));
    dst[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
  if (threadIdx.x == 0) { tc[r] = t[row]; rinv[r] = rr; }
}

// d(gain) partial of one chunk, per column, rows summed in a fixed order:
// part[h] = sum_rows dx[row, h] * xhat[row, h] (dx is the grad_hidden row the
// backward GEMM just wrote).  One block owns 32 columns.
constexpr int DG_THREADS = 256;
__global__ void __launch_bounds__(DG_THREADS)
    rmsnorm_dgain_kernel(const int* hdr, const int* __restrict__ idx, long long c0, int C, int H,
                         const uint16_t* __restrict__ X, const float* __restrict__ rinv,
                         const uint16_t* __restrict__ gh, float* __restrict__ part) {
  __shared__ float acc[DG_THREADS / 32][32];
  const int Cl = chunk_rows(hdr, c0, C);
  const int lane = threadIdx.x % 32, w = threadIdx.x / 32;
  const int h = blockIdx.x * 32 + lane;
  float a = 0.f;
  if (h < H)
    for (int r = w; r < Cl; r += DG_THREADS / 32) {
      const long long row = idx[c0 + r];
      const float dx = __uint_as_float(static_cast<uint32_t>(gh[row * H + h]) << 16);
      const float x = __uint_as_float(static_cast<uint32_t>(X[row * H + h]) << 16);
      a = fmaf(dx, x * rinv[r], a);
    }
  acc[w][lane] = a;
  __syncthreads();
  if (w == 0 && h < H) {
    float s = 0.f;
#pragma unroll
    for (int k = 0; k < DG_THREADS / 32; ++k) s += acc[k][lane];
    part[h] = s;
  }
}

// In place: grad_hidden row = r (g dx - xhat mean(g dx xhat)) (RMSNorm backward).
__global__ void __launch_bounds__(NORM_THREADS)
    rmsnorm_bwd_rows_kernel(const int* hdr, const int* __restrict__ idx, long long c0, int C, int H,
                            const uint16_t* __restrict__ X, const uint16_t* __restrict__ gain,
                            const float* __restrict__ rinv, uint16_t* __restrict__ gh) {
  __shared__ float red[NORM_THREADS / 32];
  const int r = blockIdx.x;
  const int Cl = chunk_rows(hdr, c0, C);
  if (r >= Cl) return;
  const long long row = idx[c0 + r];
  const float rr = rinv[r];
  const uint4* xs = reinterpret_cast<const uint4*>(X + row * H);
  const uint4* gs = reinterpret_cast<const uint4*>(gain);
  uint4* ds = reinterpret_cast<uint4*>(gh + row * H);
  const int n16 = H / 8;
  float dot = 0.f;
  for (int c = threadIdx.x; c < n16; c += NORM_THREADS) {
    const uint4 xw = xs[c], gw = gs[c], dw = ds[c];
    const uint32_t xq[4] = {xw.x, xw.y, xw.z, xw.w}, gq[4] = {gw.x, gw.y, gw.z, gw.w}, dq[4] = {dw.x, dw.y, dw.z, dw.w};
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      dot = fmaf(bf16_lo(gq[k]) * bf16_lo(dq[k]), bf16_lo(xq[k]) * rr, dot);
      dot = fmaf(bf16_hi(gq[k]) * bf16_hi(dq[k]), bf16_hi(xq[k]) * rr, dot);
    }
  }
  const float mean = block_reduce(dot, AddOp(), 0.f, red) / static_cast<float>(H);
  for (int c = threadIdx.x; c < n16; c += NORM_THREADS) {
    const uint4 xw = xs[c], gw = gs[c], dw = ds[c];
    const uint32_t xq[4] = {xw.x, xw.y, xw.z, xw.w}, gq[4] = {gw.x, gw.y, gw.z, gw.w}, dq[4] = {dw.x, dw.y, dw.z, dw.w};
    uint32_t o[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const float d0 = rr * (bf16_lo(gq[k]) * bf16_lo(dq[k]) - bf16_lo(xq[k]) * rr * mean);
      const float d1 = rr * (bf16_hi(gq[k]) * bf16_hi(dq[k]) - bf16_hi(xq[k]) * rr * mean);
      o[k] = ptx::pack_bf16x2(d0, d1);
    }
    ds[c] = make_uint4(o[0], o[1], o[2], o[3]);
  }
}

// grad_gain[h] = sum over chunks, in chunk order, of the chunk partials.
__global__ void dgain_reduce_kernel(const float* __restrict__ part, long long n_chunks, int H,
                                    float* __restrict__ grad_gain) {
  const int h = blockIdx.x * blockDim.x + threadIdx.x;
  if (h >= H) return;
  double s = 0.0;
  for (long long c = 0; c < n_chunks; ++c) s += part[c * H + h];
  grad_gain[h] = static_cast<float>(s);
}

// ---------------------------------------------------------------------------
// Vocabulary-parallel LM head: per-token statistics of one vocabulary shard,
// and the merge of all shards' statistics into the log-sum-exp (the online
// softmax merge of "Alisa's book of LLMs", applied across shards).
// ---------------------------------------------------------------------------

// One chunk row: max and sum exp over the shard's parts, and the target logit
// when the target lies in the shard (else 0), written at the token's row.
__global__ void __launch_bounds__(LSE_THREADS)
    shard_stats_kernel(const int* hdr, const int* __restrict__ idx, long long c0, int C, int nparts,
                       const float2* __restrict__ part, const float* __restrict__ zt, const int* __restrict__ tc,
                       float* __restrict__ row_max, float* __restrict__ row_sumexp, float* __restrict__ row_zt) {
  __shared__ float red[LSE_THREADS / 32];
  const int r = blockIdx.x;
  const int Cl = chunk_rows(hdr, c0, C);
  if (r >= Cl) return;
  const float2* pr = part + static_cast<size_t>(r) * nparts;
  float m = -INFINITY;
  for (int j = threadIdx.x; j < nparts; j += LSE_THREADS) m = fmaxf(m, pr[j].x);
  m = block_reduce(m, MaxOp(), -INFINITY, red);
  float d = 0.f;
  for (int j = threadIdx.x; j < nparts; j += LSE_THREADS) d += pr[j].y * exp2f((pr[j].x - m) * LOG2E);
  d = block_reduce(d, AddOp(), 0.f, red);
  if (threadIdx.x == 0) {
    const long long row = idx[c0 + r];
    row_max[row] = m;
    row_sumexp[row] = d;
    row_zt[row] = tc[r] >= 0 ? zt[r] : 0.f;
  }
}

// Rows of ignored tokens: max 0, sum 0, target logit 0.
__global__ void shard_stats_ignored_kernel(const int* hdr, const int* __restrict__ idx, long long N,
                                           float* row_max, float* row_sumexp, float* row_zt) {
  const long long nv = hdr[HDR_NVALID];
  for (long long i = nv + static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < N;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const long long row = idx[i];
    row_max[row] = 0.f;
    row_sumexp[row] = 0.f;
    row_zt[row] = 0.f;
  }
}

// sum exp of a shard rescaled to the global max: d *= exp(m_local - m_global)
__global__ void vocab_rescale_kernel(const float* __restrict__ m_local, const float* __restrict__ m_global,
                                     float* __restrict__ sumexp, long long N) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < N;
       i += static_cast<long long>(gridDim.x) * blockDim.x)
    sumexp[i] *= exp2f((m_local[i] - m_global[i]) * LOG2E);
}

// lse = m + log(sum), row loss = lse - z_t, loss = fixed-order sum / n_valid.
constexpr int VF_THREADS = 1024;
__global__ void __launch_bounds__(VF_THREADS)
    vocab_finish_kernel(const float* __restrict__ m, const float* __restrict__ sumexp, const float* __restrict__ zt,
                        const int* __restrict__ t, long long N, int ii, int reduce_sum, float* __restrict__ lse,
                        float* __restrict__ row_loss, float* loss, int* n_valid) {
  __shared__ double red[VF_THREADS / 32];
  __shared__ int redn[VF_THREADS / 32];
  double s = 0.0;
  int n = 0;
  for (long long i = threadIdx.x; i < N; i += VF_THREADS) {
    const bool valid = t[i] != ii;
    const float l = valid ? m[i] + logf(sumexp[i]) : 0.f;
    const float rl = valid ? l - zt[i] : 0.f;
    if (lse) lse[i] = l;
    if (row_loss) row_loss[i] = rl;
    s += rl;
    n += valid ? 1 : 0;
  }
  s = block_reduce(s, AddOp(), 0.0, red);
  n = block_reduce(n, AddOp(), 0, redn);
  if (threadIdx.x == 0) {
    *loss = n == 0 ? 0.f : static_cast<float>(reduce_sum ? s : s / static_cast<double>(n));
    if (n_valid) *n_valid = n;
  }
}

// grad_hidden (bf16) and grad_weight (fp32) times a device scalar, in place:
// the backward of the fused op when the incoming gradient of the loss is not
// one ("efficient-llm-anatomy" README: the backward pass only distributes the
// gradients computed during forward).
__global__ void scale_grads_kernel(uint16_t* __restrict__ gh, long long n8, float* __restrict__ gw, long long n4,
                                   const float* __restrict__ scale) {
  const float a = *scale;
  const long long stride = static_cast<long long>(gridDim.x) * blockDim.x;
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
    uint4 w = reinterpret_cast<uint4*>(gh)[i];
    uint32_t in[4] = {w.x, w.y, w.z, w.w};
    uint32_t out[4];
#pragma unroll
    for (int g = 0; g < 4; ++g)
      out[g] = ptx::pack_bf16x2(__uint_as_float(in[g] << 16) * a, __uint_as_float(in[g] & 0xFFFF0000u) * a);
    reinterpret_cast<uint4*>(gh)[i] = make_uint4(out[0], out[1], out[2], out[3]);
  }
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4; i += stride) {
    float4 v = reinterpret_cast<float4*>(gw)[i];
    v.x *= a; v.y *= a; v.z *= a; v.w *= a;
    reinterpret_cast<float4*>(gw)[i] = v;
  }
}

__global__ void timeout_selftest_kernel(int* hdr, unsigned long long timeout_ns) {
  __shared__ uint64_t bar;
  if (threadIdx.x != 0) return;
  hdr[HDR_STATUS] = 0;
  ptx::mbar_init(&bar, 1);
  ptx::mbar_fence_init();
  // Phase 0 of a fresh barrier completes only when someone arrives: nobody will.
  const uint64_t t0 = ptx::global_timer_ns();
  bool done = false;
  for (;;) {
    if (ptx::mbar_test(&bar, 0)) { done = true; break; }
    if (ptx::global_timer_ns() - t0 > timeout_ns) break;
  }
  if (!done) atomicOr(&hdr[HDR_STATUS], STATUS_TIMEOUT);
}

// The fp32 grad_weight accumulator rounded once to the bf16 output
// (FLCE_GW_BF16): gradients accumulate in fp32 and only the finished sum is
// stored at the parameter's precision ("Alisa's book of LLMs", "Precision").
__global__ void f32_to_bf16_kernel(const float4* __restrict__ src, long long n4, uint2* __restrict__ dst) {
  for (long long i = static_cast<long long>(blockIdx.x) * blockDim.x + threadIdx.x; i < n4;
       i += static_cast<long long>(gridDim.x) * blockDim.x) {
    const float4 v = __ldcs(src + i);
    dst[i] = make_uint2(ptx::pack_bf16x2(v.x, v.y), ptx::pack_bf16x2(v.z, v.w));
  }
}

inline int grid_for(long long work, int threads, int cap) {
  long long g = (work + threads - 1) / threads;
  if (g < 1) g = 1;
  return static_cast<int>(g < cap ? g : cap);
}

}  // namespace

cudaError_t launch_prep(const int* targets, long long N, int V, int ii, int* hdr, int* idx, int* n_valid_out,
                        int* counters, long long n_counters, cudaStream_t s) {
  prep_kernel<<<1, PREP_THREADS, 0, s>>>(targets, N, V, ii, hdr, idx, n_valid_out, counters, n_counters);
  return cudaGetLastError();
}

cudaError_t launch_zero_ignored(const int* hdr, const int* idx, long long N, long long row_bytes, void* gh,
                                cudaStream_t s) {
  zero_ignored_kernel<<<grid_for(N * (row_bytes / 16), 256, 1216), 256, 0, s>>>(hdr, idx, N, row_bytes,
                                                                                static_cast<unsigned char*>(gh));
  return cudaGetLastError();
}

cudaError_t launch_gather(const uint16_t* hidden, const int* targets, const int* hdr, const int* idx,
                          long long c0, int C, int H, uint16_t* xc, int* tc, int v0, int vs, cudaStream_t s) {
  gather_kernel<<<C, 128, 0, s>>>(hidden, targets, hdr, idx, c0, C, H, xc, tc, v0, vs);
  return cudaGetLastError();
}

cudaError_t launch_lse_dz(const int* hdr, long long c0, int C, int V, long long ldz, int nparts,
                          const float2* part, const float* zt, const int* tc, float* rl, uint16_t* z,
                          int reduce_sum, int make_dz, const float* lse_ext, const int* idx, cudaStream_t s) {
  lse_dz_kernel<<<C, LSE_THREADS, 0, s>>>(hdr, c0, C, V, ldz, nparts, part, zt, tc, rl, z, reduce_sum, make_dz,
                                          lse_ext, idx);
  return cudaGetLastError();
}

cudaError_t launch_finalize(const int* hdr, const int* idx, const float* rl, long long N, int reduce_sum,
                            float* loss, int* n_valid_out, float* row_loss, cudaStream_t s) {
  const int blocks = row_loss ? static_cast<int>(std::min<long long>((N + 4 * FIN_THREADS - 1) / (4 * FIN_THREADS), 148)) : 1;
  finalize_kernel<<<blocks, FIN_THREADS, 0, s>>>(hdr, idx, rl, N, reduce_sum, loss, n_valid_out, row_loss);
  return cudaGetLastError();
}

cudaError_t launch_gather_norm(const uint16_t* hidden, const int* targets, const int* hdr, const int* idx,
                               long long c0, int C, int H, const uint16_t* gain, float eps, uint16_t* xc, int* tc,
                               float* rinv, cudaStream_t s) {
  gather_norm_kernel<<<C, NORM_THREADS, 0, s>>>(hidden, targets, hdr, idx, c0, C, H, gain, eps, xc, tc, rinv);
  return cudaGetLastError();
}

cudaError_t launch_rmsnorm_bwd(const int* hdr, const int* idx, long long c0, int C, int H, const uint16_t* hidden,
                               const uint16_t* gain, const float* rinv, uint16_t* grad_hidden, float* dgain_partial,
                               cudaStream_t s) {
  rmsnorm_dgain_kernel<<<(H + 31) / 32, DG_THREADS, 0, s>>>(hdr, idx, c0, C, H, hidden, rinv, grad_hidden,
                                                            dgain_partial);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  rmsnorm_bwd_rows_kernel<<<C, NORM_THREADS, 0, s>>>(hdr, idx, c0, C, H, hidden, gain, rinv, grad_hidden);
  return cudaGetLastError();
}

cudaError_t launch_dgain_reduce(const float* partials, long long n_chunks, int H, float* grad_gain, cudaStream_t s) {
  dgain_reduce_kernel<<<(H + 255) / 256, 256, 0, s>>>(partials, n_chunks, H, grad_gain);
  return cudaGetLastError();
}

cudaError_t launch_shard_stats(const int* hdr, const int* idx, long long c0, int C, int nparts, const float2* part,
                               const float* zt, const int* tc, float* row_max, float* row_sumexp, float* row_zt,
                               cudaStream_t s) {
  shard_stats_kernel<<<C, LSE_THREADS, 0, s>>>(hdr, idx, c0, C, nparts, part, zt, tc, row_max, row_sumexp, row_zt);
  return cudaGetLastError();
}

cudaError_t launch_shard_stats_ignored(const int* hdr, const int* idx, long long N, float* row_max,
                                       float* row_sumexp, float* row_zt, cudaStream_t s) {
  shard_stats_ignored_kernel<<<grid_for(N, 256, 1216), 256, 0, s>>>(hdr, idx, N, row_max, row_sumexp, row_zt);
  return cudaGetLastError();
}

cudaError_t launch_vocab_rescale(const float* m_local, const float* m_global, float* sumexp, long long N,
                                 cudaStream_t s) {
  vocab_rescale_kernel<<<grid_for(N, 256, 1216), 256, 0, s>>>(m_local, m_global, sumexp, N);
  return cudaGetLastError();
}

cudaError_t launch_vocab_finish(const float* m, const float* sumexp, const float* zt, const int* t, long long N,
                                int ii, int reduce_sum, float* lse, float* row_loss, float* loss, int* n_valid,
                                cudaStream_t s) {
  vocab_finish_kernel<<<1, VF_THREADS, 0, s>>>(m, sumexp, zt, t, N, ii, reduce_sum, lse, row_loss, loss, n_valid);
  return cudaGetLastError();
}

cudaError_t launch_scale_grads(uint16_t* grad_hidden, long long n_hidden, float* grad_weight, long long n_weight,
                               const float* scale, cudaStream_t s) {
  const long long n8 = n_hidden / 8, n4 = n_weight / 4;
  scale_grads_kernel<<<grid_for(n8 > n4 ? n8 : n4, 256, 152 * 8), 256, 0, s>>>(grad_hidden, n8, grad_weight, n4, scale);
  return cudaGetLastError();
}

cudaError_t launch_f32_to_bf16(const float* src, long long n, uint16_t* dst, cudaStream_t s) {
  const long long n4 = n / 4;
  f32_to_bf16_kernel<<<grid_for(n4, 256, 152 * 8), 256, 0, s>>>(reinterpret_cast<const float4*>(src), n4,
                                                                reinterpret_cast<uint2*>(dst));
  return cudaGetLastError();
}

cudaError_t launch_timeout_selftest(int* hdr, unsigned long long timeout_ns, cudaStream_t s) {
  timeout_selftest_kernel<<<1, 32, 0, s>>>(hdr, timeout_ns);
  return cudaGetLastError();
}

}  // namespace flce
