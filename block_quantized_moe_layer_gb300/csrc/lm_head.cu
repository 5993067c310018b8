// lm_head.cu -- output norm + Q8_0 LM head for the MTP round (T <= 8 rows).
//
// logits[t, v] = sum_h w[v, h] * rmsnorm(x[t])[h], rmsnorm(u) = u / sqrt(mean(u^2) + eps).
// Each CTA first normalises the (up to 4) rows of its token group in fp32
// and turns them into 16-bit block fixed point: per 32 columns a power-of-two
// scale 2^-s and integers X with |X| <= 2^14, stored as two byte planes (low
// byte unsigned, high byte signed).  A warp then takes 2 weight rows at a
// time; lane l reads 16 consecutive int8 codes of each row per step (one
// 128-bit load; a warp load covers 512 contiguous bytes of a row) and forms
// exact integer sums with dp4a against both planes, scaled once per half
// block by d * 2^-s.  The weights are stored as int8 codes [V][H] plus fp16
// scales [V][H/32] (the serialised Q8_0 bytes, split).
#include "layer.cuh"

namespace moe {
namespace {

constexpr int kLmThreads = 512;
constexpr int kLmRows = 2;       // weight rows per warp task
constexpr int kLmTokens = 4;     // rows of x per launch (token group)

__global__ void lm_repack_kernel(const uint8_t* __restrict__ src, int8_t* __restrict__ q, __half* __restrict__ sc,
                                 int64_t nblocks) {
  const int64_t b = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (b >= nblocks) return;
  const uint8_t* s = src + b * 34;
  sc[b] = __ushort_as_half((unsigned short)(s[0] | (s[1] << 8)));
  int8_t* d = q + b * 32;
#pragma unroll
  for (int j = 0; j < 32; ++j) d[j] = (int8_t)s[2 + j];
}

template <int L>
__global__ void __launch_bounds__(kLmThreads, 1)
lm_head_kernel(const int8_t* __restrict__ q, const __half* __restrict__ sc, int V, int H, const void* x, int T,
               float eps, float* __restrict__ logits) {
  extern __shared__ __align__(16) uint8_t lsm[];
  griddep_launch_dependents();
  if (threadIdx.x == 0) {
    // constant data: start this CTA's first rows on their way to L2 while the
    // previous kernel in the stream finishes
    const int64_t r0 = (int64_t)blockIdx.x * (kLmThreads / 32) * kLmRows;
    if (r0 < V) {
      const int64_t nr = min((int64_t)(kLmThreads / 32) * kLmRows, (int64_t)V - r0);
      prefetch_l2(q + r0 * H, (uint32_t)(nr * H));
    }
  }
  griddep_wait();  // x may come from the previous kernel in the stream
  uint8_t* lo = lsm;                                          // [T][H]
  int8_t* hi = reinterpret_cast<int8_t*>(lsm + kLmTokens * H);  // [T][H]
  float* asc = reinterpret_cast<float*>(lsm + 2 * kLmTokens * H);  // [T][H/32]
  __shared__ float red[kLmTokens][kLmThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // output norm: sum of squares per row
  for (int t = 0; t < T; ++t) {
    float s = 0.f;
    for (int c = tid; c < H; c += kLmThreads) {
      float v;
      if constexpr (L == 2) v = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(x)[(int64_t)t * H + c]);
      else v = reinterpret_cast<const float*>(x)[(int64_t)t * H + c];
      s = fmaf(v, v, s);
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
    if (lane == 0) red[t][warp] = s;
  }
  __syncthreads();
  // block fixed point of the normalised rows: warp w converts blocks w, w + 16, ...
  for (int t = 0; t < T; ++t) {
    float ss = 0.f;
    for (int w = 0; w < kLmThreads / 32; ++w) ss += red[t][w];
    const float inv = 1.f / sqrtf(ss / (float)H + eps);
    for (int b = warp; b < H / 32; b += kLmThreads / 32) {
      const int c = b * 32 + lane;
      float v;
      if constexpr (L == 2) v = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(x)[(int64_t)t * H + c]);
      else v = reinterpret_cast<const float*>(x)[(int64_t)t * H + c];
      v *= inv;
      const float amax = warp_max(fabsf(v));
      int s = 0;
      if (amax > 0.f) s = max(-100, min(120, 13 - ilogbf(amax)));
      const int X = __float2int_rn(ldexpf(v, s));
      lo[t * H + c] = (uint8_t)(X & 0xFF);
      hi[t * H + c] = (int8_t)(X >> 8);
      if (lane == 0) asc[t * (H / 32) + b] = ldexpf(1.f, -s);
    }
  }
  __syncthreads();

  const int nb = H / 32;
  const int n_tasks = (V + kLmRows - 1) / kLmRows;
  for (int task = blockIdx.x * (kLmThreads / 32) + warp; task < n_tasks; task += gridDim.x * (kLmThreads / 32)) {
    const int r0 = task * kLmRows;
    float acc[kLmRows][kLmTokens];
#pragma unroll
    for (int rr = 0; rr < kLmRows; ++rr)
#pragma unroll
      for (int t = 0; t < kLmTokens; ++t) acc[rr][t] = 0.f;
#pragma unroll 4
    for (int c0 = 0; c0 < H; c0 += 512) {
      const int col = c0 + 16 * lane, blk = col >> 5;
      uint4 qv[kLmRows];
      float d[kLmRows];
#pragma unroll
      for (int rr = 0; rr < kLmRows; ++rr) {
        const int r = min(r0 + rr, V - 1);
        qv[rr] = __ldg(reinterpret_cast<const uint4*>(q + (int64_t)r * H + col));
        d[rr] = __half2float(sc[(int64_t)r * nb + blk]);
      }
#pragma unroll
      for (int t = 0; t < kLmTokens; ++t) {
        if (t < T) {
          const uint4 xl = *reinterpret_cast<const uint4*>(lo + t * H + col);
          const uint4 xh = *reinterpret_cast<const uint4*>(hi + t * H + col);
          const float a = asc[t * nb + blk];
#pragma unroll
          for (int rr = 0; rr < kLmRows; ++rr) {
            int sl = 0, sh = 0;
            sl = dp4a_su(qv[rr].x, xl.x, sl);
            sl = dp4a_su(qv[rr].y, xl.y, sl);
            sl = dp4a_su(qv[rr].z, xl.z, sl);
            sl = dp4a_su(qv[rr].w, xl.w, sl);
            sh = dp4a_ss(qv[rr].x, xh.x, sh);
            sh = dp4a_ss(qv[rr].y, xh.y, sh);
            sh = dp4a_ss(qv[rr].z, xh.z, sh);
            sh = dp4a_ss(qv[rr].w, xh.w, sh);
            acc[rr][t] = fmaf(d[rr] * a, (float)(sl + 256 * sh), acc[rr][t]);
          }
        }
      }
    }
#pragma unroll
    for (int rr = 0; rr < kLmRows; ++rr)
#pragma unroll
      for (int t = 0; t < kLmTokens; ++t) {
        float v = acc[rr][t];
#pragma unroll
        for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
        if (lane == rr * kLmTokens + t && t < T && r0 + rr < V) logits[(int64_t)t * V + r0 + rr] = v;
      }
  }
}

}  // namespace

cudaError_t lm_repack(const uint8_t* src, int8_t* q, __half* sc, int64_t nblocks, cudaStream_t st) {
  lm_repack_kernel<<<(unsigned)((nblocks + 255) / 256), 256, 0, st>>>(src, q, sc, nblocks);
  return cudaGetLastError();
}

size_t lm_smem_bytes(int H) { return (size_t)2 * kLmTokens * H + (size_t)kLmTokens * (H / 32) * 4; }

cudaError_t lm_configure(int H) {
  cudaError_t e = cudaFuncSetAttribute(lm_head_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       (int)lm_smem_bytes(H));
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(lm_head_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)lm_smem_bytes(H));
}

// Rows are processed in groups of kLmTokens (one launch per group); x is
// fp32 (x_f32) or bf16.  The arithmetic after the norm (16-bit block fixed
// point of the normalised rows, exact dp4a sums) is the same for both.
cudaError_t lm_forward(const moe_lm_head* lm, const void* x, bool x_f32, int T, float eps, float* logits,
                       cudaStream_t st) {
  const size_t esz = x_f32 ? 4 : 2;
  for (int t0 = 0; t0 < T; t0 += kLmTokens) {
    const int n = min(kLmTokens, T - t0);
    const void* xg = static_cast<const uint8_t*>(x) + (size_t)t0 * lm->H * esz;
    float* lg = logits + (int64_t)t0 * lm->V;
    cudaError_t e;
    if (!x_f32)
      e = launch_pdl(lm_head_kernel<2>, lm->num_sms, kLmThreads, lm_smem_bytes(lm->H), st, (const int8_t*)lm->q,
                     (const __half*)lm->sc, lm->V, lm->H, xg, n, eps, lg);
    else
      e = launch_pdl(lm_head_kernel<4>, lm->num_sms, kLmThreads, lm_smem_bytes(lm->H), st, (const int8_t*)lm->q,
                     (const __half*)lm->sc, lm->V, lm->H, xg, n, eps, lg);
    if (e != cudaSuccess) return e;
  }
  return cudaSuccess;
}

}  // namespace moe
