// lm_head.cu -- output norm + Q8_0 LM head for the MTP round (T <= 8 rows).
//
// logits[t, v] = sum_h w[v, h] * rmsnorm(x[t])[h], rmsnorm(u) = u / sqrt(mean(u^2) + eps).
//
// The weights are streamed like an expert's down matrix: repacked at create
// into 32-row groups of Kc-column chunks (the Q8_0 chunk layout of
// common.cuh: codes block-major, a warp's 128-bit loads of one block cover
// the 32 rows), each chunk one 1-D bulk copy into a ring of shared-memory
// stages.  Each block takes row groups blockIdx.x, blockIdx.x + gridDim.x,
// ...; its producer thread issues the first stages before the dependency
// wait (the weights are constant data), so they load while the previous
// kernel in the stream finishes.  The (up to 4) rows of x are normalised in
// fp32 and turned into 16-bit block fixed-point records once per block; the
// 8 consumer warps take the chunk's blocks w, w + 8, ... (lane = row) with
// exact dp4a sums (gemv.cuh), and their per-row partials are summed in warp
// order.  Every wait is bounded; a timeout sets the head's status word and
// the block stops.
#include "gemv.cuh"
#include "layer.cuh"

namespace moe {
namespace {

constexpr int kLmConsumerWarps = kConsumerWarps;                      // 8
constexpr int kLmThreads = (kLmConsumerWarps + 1) * 32;               // + the producer warp
constexpr int kLmTokens = 4;                                          // rows of x per launch (token group)
constexpr int kLmMaxStages = 8;
constexpr int kLmRecB = rec_bytes(2);                                 // 16-bit block fixed point
constexpr int kLmRgBatch = 8;  // row groups whose warp partials are reduced together (one barrier pair)

__global__ void lm_zero_kernel(uint8_t* __restrict__ p, int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x) p[i] = 0;
}

struct LmParams {
  const uint8_t* w;  // [n_rg][nch][chunk]
  int V, H, nch, Kc, n_rg, T, stages;
  int64_t chunk;     // bytes of one chunk
  const void* x;
  float eps;
  float* logits;     // [T][V]
  int* status;
  uint64_t timeout_ns;
};

struct LmPlan {
  int ring, recs, red, sq, bars, total;
};
__host__ __device__ inline LmPlan lm_plan(int H, int64_t chunk, int stages) {
  LmPlan p;
  p.ring = 0;
  p.recs = (int)(chunk * stages);
  p.red = p.recs + kLmTokens * (H / 32) * kLmRecB;
  p.sq = p.red + kLmRgBatch * kLmConsumerWarps * kLmTokens * 32 * 4;
  p.bars = p.sq + kLmTokens * 8 * 4;
  p.total = p.bars + 2 * kLmMaxStages * 8 + 16;
  return p;
}

__device__ inline bool lm_wait(uint64_t* bar, uint32_t parity, const LmParams& P, int site) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > P.timeout_ns) {
      if (atomicCAS(P.status, 0, kStatusTimeout) == 0) P.status[1] = site;
      return false;
    }
  }
  return true;
}

template <int LIN, int T>
__device__ void lm_consume(const LmParams& P, uint8_t* smem, const LmPlan& plan, uint64_t* full, uint64_t* empty) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint8_t* recs = smem + plan.recs;
  float* red = reinterpret_cast<float*>(smem + plan.red);
  const int nbc = P.Kc / 32;
  float acc[kGroup];
  int i = 0;  // item (row group, chunk) counter of this block
  int j = 0;  // row groups of this block so far
  // Each row group's per-warp partials go to their own slot; the slots of
  // up to kLmRgBatch row groups are summed (in warp order) behind one
  // barrier pair, so the consumers rarely stop streaming.
  auto reduce = [&](int g_last, int n) {
    consumer_sync();
    for (int u = tid; u < n * T * 32; u += kLmConsumerWarps * 32) {
      const int q = u / (T * 32), m = (u / 32) % T, l = u & 31;
      const int gq = g_last - (n - 1 - q) * (int)gridDim.x;  // the row group of slot q
      float v = 0.f;
#pragma unroll
      for (int w = 0; w < kLmConsumerWarps; ++w) v += red[((q * kLmConsumerWarps + w) * kLmTokens + m) * 32 + l];
      const int r = gq * 32 + l;
      if (r < P.V) P.logits[(int64_t)m * P.V + r] = v;
    }
    consumer_sync();
  };
  int g = blockIdx.x;
  for (; g < P.n_rg; g += gridDim.x, ++j) {
#pragma unroll
    for (int m = 0; m < kGroup; ++m) acc[m] = 0.f;
    for (int c = 0; c < P.nch; ++c, ++i) {
      const int s = i % P.stages;
      if (!lm_wait(&full[s], (uint32_t)((i / P.stages) & 1), P, 2)) return;
      gemv_chunk_m<2, T>(smem + plan.ring + (int64_t)s * P.chunk, recs + (int64_t)c * T * nbc * kLmRecB, nbc, MOE_Q8_0,
                         0, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
    }
    const int q = j % kLmRgBatch;
#pragma unroll
    for (int m = 0; m < T; ++m) red[((q * kLmConsumerWarps + warp) * kLmTokens + m) * 32 + lane] = acc[m];
    if (q == kLmRgBatch - 1) reduce(g, kLmRgBatch);
  }
  if (j % kLmRgBatch) reduce(g - (int)gridDim.x, j % kLmRgBatch);
}

template <int LIN>
__global__ void __launch_bounds__(kLmThreads, 1) lm_stream_kernel(const __grid_constant__ LmParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const LmPlan plan = lm_plan(P.H, P.chunk, P.stages);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + plan.bars);
  uint64_t* empty = full + kLmMaxStages;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int n_items = (P.n_rg - (int)blockIdx.x + (int)gridDim.x - 1) / (int)gridDim.x * P.nch;
  griddep_launch_dependents();
  if (tid == 0) {
    for (int s = 0; s < P.stages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kLmConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();
  const bool producer = warp == kLmConsumerWarps && lane == 0;
  const uint64_t wpol = l2_evict_first_policy();
  // item i of this block: row group blockIdx.x + (i / nch) * gridDim.x, chunk i % nch
  auto issue = [&](int i) {
    const int s = i % P.stages;
    const int g = blockIdx.x + (i / P.nch) * gridDim.x, c = i % P.nch;
    mbar_arrive_expect_tx(&full[s], (uint32_t)P.chunk);
    bulk_g2s_hint(smem + plan.ring + (int64_t)s * P.chunk, P.w + ((int64_t)g * P.nch + c) * P.chunk, (uint32_t)P.chunk,
                  &full[s], wpol);
  };
  int issued = 0;
  if (producer)  // constant data: the first stages load while the previous kernel finishes
    for (; issued < min(P.stages, n_items); ++issued) issue(issued);
  griddep_wait();  // x may come from the previous kernel in the stream

  if (producer) {
    bool ok = true;
    for (; issued < n_items && ok; ++issued) {
      ok = lm_wait(&empty[issued % P.stages], (uint32_t)((issued / P.stages - 1) & 1), P, 1);
      if (ok) issue(issued);
    }
    // every copy issued has landed before the block leaves
    for (int j = max(0, issued - P.stages); j < issued; ++j)
      lm_wait(&full[j % P.stages], (uint32_t)((j / P.stages) & 1), P, 3);
  } else if (warp < kLmConsumerWarps) {
    // records of the normalised rows, [chunk][token][block] (consumers only)
    float* sq = reinterpret_cast<float*>(smem + plan.sq);  // [T][8]
    for (int t = 0; t < P.T; ++t) {
      float ss = 0.f;
      for (int c = tid; c < P.H; c += kLmConsumerWarps * 32) {
        float v;
        if constexpr (LIN == 2) v = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(P.x)[(int64_t)t * P.H + c]);
        else v = reinterpret_cast<const float*>(P.x)[(int64_t)t * P.H + c];
        ss = fmaf(v, v, ss);
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) sq[t * 8 + warp] = ss;
    }
    consumer_sync();
    const int nbc = P.Kc / 32;
    float inv[kLmTokens];
#pragma unroll
    for (int t = 0; t < kLmTokens; ++t) {
      float ss = 0.f;
      if (t < P.T)
        for (int w = 0; w < kLmConsumerWarps; ++w) ss += sq[t * 8 + w];
      inv[t] = 1.f / sqrtf(ss / (float)P.H + P.eps);
    }
    // one thread per record (t, block): the block's 32 values of row t,
    // times the row's 1/rms, into the record (no warp reductions)
    const int nb = P.H / 32;
    for (int u = tid; u < P.T * nb; u += kLmConsumerWarps * 32) {
      const int t = u / nb, b = u - t * nb;
      float v[32];
      const uint4* src = reinterpret_cast<const uint4*>(static_cast<const uint8_t*>(P.x) +
                                                        ((int64_t)t * P.H + (int64_t)b * 32) * (LIN == 2 ? 2 : 4));
      float sc = inv[0];
#pragma unroll
      for (int m = 1; m < kLmTokens; ++m)
        if (t == m) sc = inv[m];
#pragma unroll
      for (int q = 0; q < (LIN == 2 ? 4 : 8); ++q) {
        const uint4 w4 = src[q];
        if constexpr (LIN == 2) {
          const uint32_t w[4] = {w4.x, w4.y, w4.z, w4.w};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            v[8 * q + 2 * k] = __uint_as_float(w[k] << 16) * sc;
            v[8 * q + 2 * k + 1] = __uint_as_float(w[k] & 0xFFFF0000u) * sc;
          }
        } else {
          v[4 * q] = __uint_as_float(w4.x) * sc;
          v[4 * q + 1] = __uint_as_float(w4.y) * sc;
          v[4 * q + 2] = __uint_as_float(w4.z) * sc;
          v[4 * q + 3] = __uint_as_float(w4.w) * sc;
        }
      }
      const int c = b / nbc, lb = b - c * nbc;
      record_from_values<2>(v, smem + plan.recs + (((int64_t)c * P.T + t) * nbc + lb) * kLmRecB);
    }
    consumer_sync();
    switch (P.T) {
      case 1: lm_consume<LIN, 1>(P, smem, plan, full, empty); break;
      case 2: lm_consume<LIN, 2>(P, smem, plan, full, empty); break;
      case 3: lm_consume<LIN, 3>(P, smem, plan, full, empty); break;
      default: lm_consume<LIN, 4>(P, smem, plan, full, empty); break;
    }
  }
}

}  // namespace

cudaError_t repack_matrix(int fmt, const uint8_t* src, uint8_t* dst, int rows, int K, int rows_per_tile, int lr_off,
                          Chunking ch, cudaStream_t st);

// Bytes of the repacked head: ceil(V / 32) row groups of nch chunks.
size_t lm_weight_bytes(int V, int H, Chunking ch) {
  return (size_t)((V + 31) / 32) * ch.n * (size_t)chunk_bytes(MOE_Q8_0, ch.Kc);
}

// Chunking of the head's rows: chunks of at most 2048 columns (8 blocks per
// consumer warp per stage), as large as two stages beside the records allow.
Chunking lm_chunking(int H) { return choose_chunking(MOE_Q8_0, H, 0); }

cudaError_t lm_repack(const uint8_t* src, uint8_t* dst, int V, int H, cudaStream_t st) {
  const Chunking ch = lm_chunking(H);
  const int64_t n = (int64_t)lm_weight_bytes(V, H, ch);
  lm_zero_kernel<<<(unsigned)std::min<int64_t>((n + 255) / 256, 4096), 256, 0, st>>>(dst, n);  // rows past V
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  return repack_matrix(MOE_Q8_0, src, dst, V, H, 32, 0, ch, st);
}

namespace {
int lm_stages(int H, int64_t chunk, int max_optin) {
  int s = kLmMaxStages;
  while (s > 2 && lm_plan(H, chunk, s).total > max_optin) --s;
  return s;
}
}  // namespace

cudaError_t lm_configure(int H, int max_optin) {
  const Chunking ch = lm_chunking(H);
  const int64_t chunk = chunk_bytes(MOE_Q8_0, ch.Kc);
  const int bytes = lm_plan(H, chunk, lm_stages(H, chunk, max_optin)).total;
  cudaError_t e = cudaFuncSetAttribute(lm_stream_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(lm_stream_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
}

// Rows are processed in groups of kLmTokens (one launch per group); x is
// fp32 (x_f32) or bf16.  The arithmetic after the norm (16-bit block fixed
// point of the normalised rows, exact dp4a sums) is the same for both.
cudaError_t lm_forward(const moe_lm_head* lm, const void* x, bool x_f32, int T, float eps, float* logits,
                       cudaStream_t st) {
  const size_t esz = x_f32 ? 4 : 2;
  const Chunking ch = lm_chunking(lm->H);
  LmParams P{};
  P.w = lm->w;
  P.V = lm->V;
  P.H = lm->H;
  P.nch = ch.n;
  P.Kc = ch.Kc;
  P.n_rg = (lm->V + 31) / 32;
  P.chunk = chunk_bytes(MOE_Q8_0, ch.Kc);
  P.stages = lm_stages(lm->H, P.chunk, lm->max_optin);
  P.eps = eps;
  P.status = lm->status;
  P.timeout_ns = 2000000000ull;
  const int smem = lm_plan(lm->H, P.chunk, P.stages).total;
  for (int t0 = 0; t0 < T; t0 += kLmTokens) {
    P.T = min(kLmTokens, T - t0);
    P.x = static_cast<const uint8_t*>(x) + (size_t)t0 * lm->H * esz;
    P.logits = logits + (int64_t)t0 * lm->V;
    cudaError_t e;
    if (!x_f32) e = launch_pdl(lm_stream_kernel<2>, lm->num_sms, kLmThreads, smem, st, P);
    else e = launch_pdl(lm_stream_kernel<4>, lm->num_sms, kLmThreads, smem, st, P);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
