// repack.cu -- serialised weights -> the device layouts the kernels stream.
//
// A matrix [rows, K] is cut into tiles of `rows_per_tile` rows; tile t's
// rows land at rows lr_off .. lr_off + rows_per_tile - 1 of 32-row chunks
// (gate rows at chunk rows 0-15 and up rows at 16-31 of the same gate/up
// tile, so that one tile yields complete SwiGLU outputs).  Each (tile, chunk)
// is contiguous: chunk_bytes(fmt, Kc) at offset (tile * nch + c) * chunk_bytes.
// Within a chunk the 16-byte pieces of the 32 rows of one block are adjacent,
// so the 32 lanes of a warp (one row each) read one block with conflict-free
// 128-bit loads.
#include "common.cuh"

namespace moe {

// Q8_0: one thread per (row, 32-weight block).
__global__ void repack_q8_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int rows, int K,
                                 int rows_per_tile, int lr_off, int nch, int Kc) {
  const int nb = K / 32;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)rows * nb) return;
  const int r = (int)(i / nb), b = (int)(i % nb);
  const int tile = r / rows_per_tile, lr = r % rows_per_tile + lr_off;
  const int nbc = Kc / 32, c = b / nbc, lb = b % nbc;
  const int64_t cb = chunk_bytes(MOE_Q8_0, Kc);
  uint8_t* chunk = dst + ((int64_t)tile * nch + c) * cb;
  const uint8_t* s = src + i * 34;
  uint8_t* q0 = chunk + ((int64_t)(lb * 2 + 0) * kRows + lr) * 16;
  uint8_t* q1 = chunk + ((int64_t)(lb * 2 + 1) * kRows + lr) * 16;
#pragma unroll
  for (int j = 0; j < 16; ++j) {
    q0[j] = s[2 + j];
    q1[j] = s[18 + j];
  }
  uint8_t* sc = chunk + nbc * 1024 + (lb * kRows + lr) * 2;
  sc[0] = s[0];
  sc[1] = s[1];
}

// Q4KS: one thread per (row, 256-weight superblock).
__global__ void repack_q4ks_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int rows, int K,
                                   int rows_per_tile, int lr_off, int nch, int Kc) {
  const int ns = K / 256;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)rows * ns) return;
  const int r = (int)(i / ns), sb = (int)(i % ns);
  const int tile = r / rows_per_tile, lr = r % rows_per_tile + lr_off;
  const int nbc = Kc / 32;                     // sub-blocks per chunk
  const int c = (sb * 8) / nbc, lsb0 = (sb * 8) % nbc;
  const int64_t cb = chunk_bytes(MOE_Q4KS, Kc);
  uint8_t* chunk = dst + ((int64_t)tile * nch + c) * cb;
  const uint8_t* s = src + i * 144;
  uint8_t* hdr = chunk + nbc * 512 + ((lsb0 / 8) * kRows + lr) * 16;
#pragma unroll
  for (int j = 0; j < 16; ++j) hdr[j] = s[j];
  for (int j = 0; j < 8; ++j) {
    // codes of sub-block j in weight order
    uint8_t q[32];
#pragma unroll
    for (int l = 0; l < 16; ++l) {
      const uint8_t v = s[16 + 16 * j + l];
      q[2 * l] = v & 0x0F;
      q[2 * l + 1] = v >> 4;
    }
    uint8_t* out = chunk + ((int64_t)(lsb0 + j) * kRows + lr) * 16;
#pragma unroll
    for (int w = 0; w < 4; ++w)
#pragma unroll
      for (int bb = 0; bb < 4; ++bb) out[4 * w + bb] = (uint8_t)(q[8 * w + bb] | (q[8 * w + 4 + bb] << 4));
  }
}

// Router fp32 [E, H] -> [E_pad/32][H/256][64 float4 columns][32 rows][4].
__global__ void repack_router_kernel(const float* __restrict__ src, float4* __restrict__ dst, int E, int E_pad,
                                     int H) {
  const int n4 = H / 4;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)E_pad * n4) return;
  const int r = (int)(i / n4), c4 = (int)(i % n4);
  const int rg = r / 32, lr = r % 32, ks = c4 / 64, k4 = c4 % 64;
  const int n_ks = H / kRouterKc;
  float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
  if (r < E) v = *reinterpret_cast<const float4*>(src + (int64_t)r * H + 4 * c4);
  dst[(((int64_t)rg * n_ks + ks) * 64 + k4) * 32 + lr] = v;
}

cudaError_t repack_matrix(int fmt, const uint8_t* src, uint8_t* dst, int rows, int K, int rows_per_tile,
                          int lr_off, Chunking ch, cudaStream_t st) {
  const int threads = 256;
  if (fmt == MOE_Q8_0) {
    const int64_t n = (int64_t)rows * (K / 32);
    repack_q8_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, st>>>(src, dst, rows, K, rows_per_tile,
                                                                                   lr_off, ch.n, ch.Kc);
  } else if (fmt == MOE_Q4KS) {
    const int64_t n = (int64_t)rows * (K / 256);
    repack_q4ks_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, st>>>(src, dst, rows, K,
                                                                                     rows_per_tile, lr_off, ch.n,
                                                                                     ch.Kc);
  } else {
    return cudaErrorInvalidValue;
  }
  return cudaGetLastError();
}

cudaError_t repack_router(const float* src, float* dst, int E, int E_pad, int H, cudaStream_t st) {
  const int64_t n = (int64_t)E_pad * (H / 4);
  repack_router_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(src, reinterpret_cast<float4*>(dst), E, E_pad,
                                                                     H);
  return cudaGetLastError();
}

}  // namespace moe
