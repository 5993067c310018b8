// quantize.cu -- fp32 -> serialised Q8_0 / Q4KS, bit-exact and deterministic.
//
// The formats are the library's readings of the Q8_0 and Q4_K types the
// pages name ("Step-5 Preview GGUF", "Precision distribution" table; "Step
// 3.7 Flash Mixed-Quant GGUF", "Tensor recipe" table).  Every step rounds
// exactly once in IEEE fp32 (the __f*_rn intrinsics keep the compiler from
// fusing them), so the bytes do not depend on the compiler or the GPU.
#include "common.cuh"

namespace moe {

__device__ __forceinline__ float round_half_away(float v) { return roundf(v); }

// One thread per 32-weight block.  A serialised block is 34 bytes, so it is
// written as 17 aligned 16-bit words (the scale, then 16 pairs of codes).
__global__ void quantize_q8_kernel(const float* __restrict__ w, uint8_t* __restrict__ out, int64_t nblocks) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nblocks) return;
  const float* s = w + i * 32;
  float amax = 0.f;
#pragma unroll
  for (int j = 0; j < 32; ++j) amax = fmaxf(amax, fabsf(s[j]));
  const float d = __fdiv_rn(amax, 127.f);
  uint16_t* o = reinterpret_cast<uint16_t*>(out + i * 34);
  o[0] = __half_as_ushort(__float2half_rn(d));
#pragma unroll
  for (int j = 0; j < 32; j += 2) {
    uint32_t pair = 0;
#pragma unroll
    for (int u = 0; u < 2; ++u) {
      int q = 0;
      if (d > 0.f) q = (int)fminf(127.f, fmaxf(-127.f, round_half_away(__fdiv_rn(s[j + u], d))));
      pair |= ((uint32_t)q & 0xFFu) << (8 * u);
    }
    o[1 + j / 2] = (uint16_t)pair;
  }
}

__global__ void quantize_q4ks_kernel(const float* __restrict__ w, uint8_t* __restrict__ out, int64_t nsuper) {
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= nsuper) return;
  const float* s = w + i * 256;
  float A[8], B[8];
  float maxA = 0.f, maxB = 0.f;
  for (int sb = 0; sb < 8; ++sb) {
    float lo = 0.f, hi = -INFINITY;
    for (int j = 0; j < 32; ++j) {
      const float v = s[sb * 32 + j];
      lo = fminf(lo, v);
      hi = fmaxf(hi, v);
    }
    A[sb] = __fdiv_rn(__fsub_rn(hi, lo), 15.f);
    B[sb] = __fsub_rn(0.f, lo);
    maxA = fmaxf(maxA, A[sb]);
    maxB = fmaxf(maxB, B[sb]);
  }
  const __half dh = __float2half_rn(__fdiv_rn(maxA, 63.f));
  const __half mh = __float2half_rn(__fdiv_rn(maxB, 63.f));
  const float dF = __half2float(dh), mF = __half2float(mh);
  int sc[8], mm[8];
  for (int sb = 0; sb < 8; ++sb) {
    sc[sb] = dF > 0.f ? (int)fminf(63.f, fmaxf(0.f, round_half_away(__fdiv_rn(A[sb], dF)))) : 0;
    mm[sb] = mF > 0.f ? (int)fminf(63.f, fmaxf(0.f, round_half_away(__fdiv_rn(B[sb], mF)))) : 0;
  }
  // header and codes are assembled in registers and stored as 16-byte words
  // (a serialised superblock is 144 bytes, so each one starts 16-byte aligned)
  uint32_t words[3] = {0u, 0u, 0u};  // sixteen 6-bit fields, little-endian bit stream
  for (int f = 0; f < 16; ++f) {
    const uint32_t v = (uint32_t)(f < 8 ? sc[f] : mm[f - 8]);
    const int p = 6 * f, wi = p >> 5, sh = p & 31;
    words[wi] |= v << sh;
    if (sh > 26) words[wi + 1] |= v >> (32 - sh);
  }
  uint4* o = reinterpret_cast<uint4*>(out + i * 144);
  o[0] = make_uint4((uint32_t)__half_as_ushort(dh) | ((uint32_t)__half_as_ushort(mh) << 16), words[0], words[1],
                    words[2]);
  for (int sb = 0; sb < 8; ++sb) {
    const float a = __fmul_rn(dF, (float)sc[sb]);
    const float bq = __fmul_rn(mF, (float)mm[sb]);
    uint32_t qw[4] = {0u, 0u, 0u, 0u};  // 16 bytes = 32 codes of this sub-block
    for (int j = 0; j < 32; ++j) {
      const float v = s[sb * 32 + j];
      const int q = a > 0.f ? (int)fminf(15.f, fmaxf(0.f, round_half_away(__fdiv_rn(__fadd_rn(v, bq), a)))) : 0;
      qw[j >> 3] |= (uint32_t)q << (4 * (j & 7));  // weight j: byte j/2, low nibble for even j
    }
    o[1 + sb] = make_uint4(qw[0], qw[1], qw[2], qw[3]);
  }
}

cudaError_t quantize_launch(int fmt, const float* w, int64_t rows, int64_t cols, void* out, cudaStream_t st) {
  if (fmt == MOE_Q8_0) {
    const int64_t n = rows * (cols / 32);
    quantize_q8_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(w, static_cast<uint8_t*>(out), n);
  } else if (fmt == MOE_Q4KS) {
    const int64_t n = rows * (cols / 256);
    quantize_q4ks_kernel<<<(unsigned)((n + 127) / 128), 128, 0, st>>>(w, static_cast<uint8_t*>(out), n);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

}  // namespace moe
