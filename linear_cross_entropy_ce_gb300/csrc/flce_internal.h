// Internal declarations shared by the CUDA translation units of libflce.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace flce {

// Device status word bits (workspace header word 0).
constexpr int STATUS_BADTARGET = 1;
constexpr int STATUS_TIMEOUT = 2;

// Workspace header words.
constexpr int HDR_STATUS = 0;
constexpr int HDR_NVALID = 1;
constexpr int HDR_STALL = 2;   // first pipeline wait that timed out: site | rank << 8 | block << 12
constexpr int HDR_STALL_COUNT = 3;   // number of timed-out waits
constexpr int HDR_STALL_LOG = 8;     // up to 8 records (code, detail) of timed-out waits
constexpr int STALL_LOG_MAX = 8;
constexpr int HDR_WORDS = 64;

// GEMM tile shape: a CTA pair (cluster of 2, tcgen05 cta_group::2) owns a
// 256 x 256 fp32 accumulator, 128 rows in each CTA's TMEM, and streams K in
// blocks of 64 bf16 (one 128-byte swizzle row).  BM is the rows per CTA.
constexpr int BM = 128;
constexpr int PAIR_M = 2 * BM;
constexpr int BN = 256;
constexpr int BK = 64;
// The logits epilogue keeps one (max, sum exp) pair per row and 128-column
// vocabulary part (each epilogue warpgroup owns half of a 256-column tile).
constexpr int PART_COLS = 128;

enum GemmMode : int {
  MODE_LOGITS = 0,  // z = Xc W^T, epilogue: per 128-column part (max, sum exp), z_t, shifted bf16 logits
  MODE_BWD = 1,     // one launch holding both consumers of dz:
                    //   grad_hidden rows = dz W          (units [0, n_dx))
                    //   grad_weight (+)= dz^T Xc         (units [n_dx, n_dx + n_dw))
};

struct GemmArgs {
  int mode;
  const int* hdr;       // workspace header (n_valid lives in HDR_NVALID)
  int* status;          // workspace header word HDR_STATUS
  int* counter;         // dynamic tile counter of this launch (zero before it)
  long long c0;         // first compacted row of this chunk
  int C;                // chunk capacity (rows)
  int H, V;
  long long ldz;        // row stride (elements) of the chunk logits buffer
  int nvt;              // vocabulary tiles: ceil(V / BN)
  int nparts;           // vocabulary parts: ceil(V / PART_COLS)
  int store_z;          // LOGITS: write the shifted bf16 logits
  int accumulate;       // BWD: add into grad_weight (chunks after the first)
  int first_chunk;      // BWD: chunk 0 (writes zeros when it is empty)
  int splits;           // BWD: vocabulary splits of the grad_hidden GEMM
  int kb_per_split;     // BWD: K blocks per split
  int interleave;       // BWD: spread the dX units through the dW units (else dX units first)
  int pf_threads;       // BWD, accumulating: the epilogue threads prefetch the grad_weight tile into L2
                        // (else one TMA prefetch when the tile's main loop starts)
  int* flags;           // BWD, splits > 1: per (tile, CTA, warpgroup) count of finished splits (zero before)
  unsigned long long timeout_ns;
  int debug_stall;      // test hook: the MMA issuer withholds the accumulator-ready signal of each
                        // pair's first unit, so that the epilogue's bounded wait runs out
  // epilogue operands
  uint16_t* z;          // [C][ldz] bf16
  float2* part;         // [C][nparts] (part max, part sum of exp)
  float* zt;            // [C] target logit
  const int* tc;        // [C] chunk targets (-1 for padding rows)
  const int* idx;       // [N] compacted row -> token row
  uint16_t* grad_hidden;// [N][H] bf16
  float* grad_hidden_f32; // [N][H] fp32 instead of grad_hidden when not null (vocabulary shards)
  float* grad_weight;   // [V][H] fp32 (zero fill of an empty first chunk)
  const float* dxacc;   // [C][H] fp32 sum of the grad_hidden splits (splits > 1)
};

// Tensor maps of one launch.  LOGITS: a0 = Xc (K-major), b0 = W (K-major).
// BWD: a0 = dz (K-major), b0 = W (MN-major), a1 = dz (MN-major view),
// b1 = Xc (MN-major), out = grad_weight (fp32, store / reduce-add of 16 x 128
// slices), pf = grad_weight again with a 256 x 128 box for L2 prefetches.
struct GemmMaps {
  CUtensorMap a0, b0, a1, b1, out;
};

int gemm_smem_bytes();
cudaError_t gemm_prepare(int device);
cudaError_t gemm_max_pairs(int* pairs);   // CTA pairs resident at once (current device)
cudaError_t launch_gemm(const GemmArgs& a, const GemmMaps& m, int grid, cudaStream_t s);

// Elementwise / bookkeeping kernels (flce_aux.cu).
cudaError_t launch_prep(const int* targets, long long N, int V, int ignore_index,
                        int* hdr, int* idx, int* n_valid_out, int* counters, long long n_counters,
                        cudaStream_t s);
cudaError_t launch_zero_ignored(const int* hdr, const int* idx, long long N, long long row_bytes,
                                void* grad_hidden, cudaStream_t s);
cudaError_t launch_gather(const uint16_t* hidden, const int* targets, const int* hdr,
                          const int* idx, long long c0, int C, int H,
                          uint16_t* xc, int* tc, int v0, int vs, cudaStream_t s);
cudaError_t launch_lse_dz(const int* hdr, long long c0, int C, int V, long long ldz,
                          int nparts, const float2* part, const float* zt, const int* tc,
                          float* rl, uint16_t* z, int reduce_sum, int make_dz,
                          const float* lse_ext, const int* idx, cudaStream_t s);
cudaError_t launch_finalize(const int* hdr, const int* idx, const float* rl,
                            long long N, int reduce_sum, float* loss, int* n_valid_out,
                            float* row_loss, cudaStream_t s);
// Final RMSNorm fused in front of the LM head.
cudaError_t launch_gather_norm(const uint16_t* hidden, const int* targets, const int* hdr, const int* idx,
                               long long c0, int C, int H, const uint16_t* gain, float eps, uint16_t* xc,
                               int* tc, float* rinv, cudaStream_t s);
cudaError_t launch_rmsnorm_bwd(const int* hdr, const int* idx, long long c0, int C, int H,
                               const uint16_t* hidden, const uint16_t* gain, const float* rinv,
                               uint16_t* grad_hidden, float* dgain_partial, cudaStream_t s);
cudaError_t launch_dgain_reduce(const float* partials, long long n_chunks, int H, float* grad_gain,
                                cudaStream_t s);
// Vocabulary-parallel LM head.
cudaError_t launch_shard_stats(const int* hdr, const int* idx, long long c0, int C, int nparts,
                               const float2* part, const float* zt, const int* tc, float* row_max,
                               float* row_sumexp, float* row_zt, cudaStream_t s);
cudaError_t launch_shard_stats_ignored(const int* hdr, const int* idx, long long N, float* row_max,
                                       float* row_sumexp, float* row_zt, cudaStream_t s);
cudaError_t launch_vocab_rescale(const float* m_local, const float* m_global, float* sumexp, long long N,
                                 cudaStream_t s);
cudaError_t launch_vocab_finish(const float* m, const float* sumexp, const float* zt, const int* t, long long N,
                                int ii, int reduce_sum, float* lse, float* row_loss, float* loss, int* n_valid,
                                cudaStream_t s);
cudaError_t launch_scale_grads(uint16_t* grad_hidden, long long n_hidden, float* grad_weight,
                               long long n_weight, const float* scale, cudaStream_t s);
cudaError_t launch_timeout_selftest(int* hdr, unsigned long long timeout_ns,
                                    cudaStream_t s);
// fp32 -> bf16 (round to nearest even), n a multiple of 4, both 16-byte aligned
cudaError_t launch_f32_to_bf16(const float* src, long long n, uint16_t* dst, cudaStream_t s);

}  // namespace flce
