// large_t.cu -- the layer for prefill-sized batches (T > 8).
//
// The steps of the layer (router, top-k and gates, permutation, SwiGLU
// experts, combine; see the layer definition in moe_layer.h) run as a
// sequence of launches on the caller's stream:
//   1. lt_prep    : x -> token tiles of the shared expert / router (fp16 MMA
//                   operand image), the work lists that need no routing;
//   2. GEMM       : router logits (three scaled fp16 planes of the fp32
//                   router, so the logits keep fp32 accuracy) + shared-expert
//                   gate/up;
//   3. lt_topk    : per token top-k (descending, ties to the lower index) and
//                   renormalised gates;
//   4. lt_perm    : histogram, scan, stable scatter -> offsets, perm, pos,
//                   routed token tiles and the remaining work lists;
//   5. lt_gather  : routed token tiles' activations (fp16 operand image);
//   6. GEMM       : routed gate/up + SwiGLU;
//   7. GEMM       : routed and shared down projections -> z (bf16);
//   8. lt_combine : y[t] = sum_j g[t,j] z[pos[t,j]] + z[shared t], in slot order.
// No step depends on atomics for its result; every result is deterministic.
#include <algorithm>

#include "large_t.cuh"

namespace moe {

struct LtState {
  // weights in the LT layout
  uint8_t* gu = nullptr;
  uint8_t* dn = nullptr;
  uint8_t* sgu = nullptr;
  uint8_t* sdn = nullptr;
  uint8_t* router = nullptr;
  int64_t gu_stride = 0, dn_stride = 0, router_plane = 0;
  size_t weight_bytes = 0;
  int E_pad128 = 0, Imax = 0, max_tiles = 0, max_rows = 0;
  // workspace
  void* ws = nullptr;
  size_t ws_bytes = 0;
  int* counters = nullptr;  // [0..2] queues, [3..5] exit counters, [6..8] item counts, [9] routed tiles
  int* status = nullptr;    // [4]
  float* logits = nullptr;  // [planes][T_max][E_pad128]
  int* ids = nullptr;
  uint32_t* bits = nullptr;  // [E][ceil(T_max/32)] tokens that chose each expert (one bit per token)
  float* gates = nullptr;
  int* pos = nullptr;
  int* perm = nullptr;
  int* offsets = nullptr;
  LtTile* tiles = nullptr;
  uint8_t* xg = nullptr;
  uint8_t* h = nullptr;
  __nv_bfloat16* z = nullptr;
};

namespace {

__host__ __device__ inline int round16(int v) { return (v + 15) & ~15; }

// ---------------------------------------------------------------------------
// Weight repacking into the LT layout (create time)
// ---------------------------------------------------------------------------

// Source row `o` of a [rows, K] matrix -> (row tile, tile row).
//   mode 0: down (128 rows per tile); mode 1: gate; mode 2: up.
__device__ __forceinline__ void lt_row(int mode, int o, int& rt, int& r) {
  if (mode == 0) {
    rt = o / 128;
    r = o % 128;
  } else {
    rt = o / 64;
    const int rem = o % 64;
    r = 32 * (rem / 16) + rem % 16 + (mode == 2 ? 16 : 0);
  }
}

__global__ void lt_repack_q8_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int rows, int K,
                                    int mode) {
  const int nb = K / 32;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)rows * nb) return;
  const int o = (int)(i / nb), b = (int)(i % nb);
  int rt, r;
  lt_row(mode, o, rt, r);
  const int kb = b / 2, h = b % 2;
  uint8_t* chunk = dst + rt * lt_tile_bytes(MOE_Q8_0, K) + (int64_t)kb * kLtQ8Chunk;
  const uint8_t* s = src + i * 34;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    uint8_t* q = chunk + ((h * 2 + p) * 128 + r) * 16;
#pragma unroll
    for (int j = 0; j < 16; ++j) q[j] = s[2 + 16 * p + j] ^ 0x80;  // u = q + 128 (sign bit flipped)
  }
  chunk[8192 + (h * 128 + r) * 2] = s[0];
  chunk[8192 + (h * 128 + r) * 2 + 1] = s[1];
}

__global__ void lt_repack_q4ks_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int rows, int K,
                                      int mode) {
  const int ns = K / 256;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)rows * ns) return;
  const int o = (int)(i / ns), sb = (int)(i % ns);
  int rt, r;
  lt_row(mode, o, rt, r);
  uint8_t* sup = dst + rt * lt_tile_bytes(MOE_Q4KS, K) + (int64_t)sb * kLtQ4Super;
  const uint8_t* s = src + i * 144;
#pragma unroll
  for (int j = 0; j < 16; ++j) sup[r * 16 + j] = s[j];
  for (int sub = 0; sub < 8; ++sub) {
    uint8_t* c = sup + kLtQ4Hdr + (sub / 2) * kLtQ4Codes + ((sub % 2) * 128 + r) * 16;
#pragma unroll
    for (int j = 0; j < 16; ++j) c[j] = s[16 + 16 * sub + j];
  }
}

// fp32 router [E, H] -> three fp16 planes, each holding the previous ones'
// remainder scaled by 2^11 so that it stays a normal fp16 number:
//   W1 = fp16(W), W2 = fp16(2^11 (W - W1)), W3 = fp16(2^11 (2^11 (W - W1) - W2)),
// W = W1 + 2^-11 W2 + 2^-22 W3 up to fp32's own precision (33 bits kept; each
// remainder is exact in fp32); rows zero-padded to E_pad128, LT 16-bit layout.
__global__ void lt_repack_router_kernel(const float* __restrict__ src, uint8_t* __restrict__ dst, int E, int E_pad,
                                        int H, int64_t plane_bytes) {
  const int n8 = H / 8;
  const int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (int64_t)E_pad * n8) return;
  const int row = (int)(i / n8), g = (int)(i % n8);
  const int k0 = g * 8, kb = k0 / 64, h = (k0 % 64) / 32, pc = (k0 % 32) / 8;
  const int rt = row / 128, r = row % 128;
  const int64_t off = rt * lt_tile_bytes(MOE_BF16, H) + (int64_t)kb * kLtBf16Chunk + ((h * 4 + pc) * 128 + r) * 16;
  uint32_t w[3][4];
#pragma unroll
  for (int j = 0; j < 8; j += 2) {
    float v0 = row < E ? src[(int64_t)row * H + k0 + j] : 0.f;
    float v1 = row < E ? src[(int64_t)row * H + k0 + j + 1] : 0.f;
#pragma unroll
    for (int pl = 0; pl < 3; ++pl) {
      const __half b0 = __float2half_rn(v0), b1 = __float2half_rn(v1);
      w[pl][j / 2] = (uint32_t)__half_as_ushort(b0) | ((uint32_t)__half_as_ushort(b1) << 16);
      v0 = (v0 - __half2float(b0)) * 2048.f;
      v1 = (v1 - __half2float(b1)) * 2048.f;
    }
  }
#pragma unroll
  for (int pl = 0; pl < 3; ++pl)
    *reinterpret_cast<uint4*>(dst + pl * plane_bytes + off) = make_uint4(w[pl][0], w[pl][1], w[pl][2], w[pl][3]);
}

// ---------------------------------------------------------------------------
// Forward kernels
// ---------------------------------------------------------------------------

// 8 bf16 values -> 8 fp16 values (exact for |v| in fp16's normal range;
// round to nearest otherwise)
__device__ __forceinline__ uint4 bf16x8_to_f16x8(uint4 v) {
  uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const __half2 h = __floats2half2_rn(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xFFFF0000u));
    w[i] = *reinterpret_cast<const uint32_t*>(&h);
  }
  return make_uint4(w[0], w[1], w[2], w[3]);
}

struct PrepParams {
  const __nv_bfloat16* x;
  int T, H, k, n_sh, n_items1;
  LtTile* tiles;
  int* counters;
  uint8_t* xg;
  uint32_t* bits;  // [E][ceil(T/32)], zeroed here for lt_topk
  int n_bits;
};

constexpr int kColSlices = 8;  // column slices per token tile in the operand-image kernels
constexpr int kImgSub = 16;    // 16-byte chunks per pass of an operand-image block's shared tile

// One column slice (16-byte chunks [c0, c0 + nc)) of an fp16 operand image:
// dst[c][r] for r < n_pad (rows past n zero), row r read from row(r).  Each
// pass goes through a shared tile [kLtMaxN][kImgSub + 1] (the pad keeps the
// transposed reads free of bank conflicts), so that the loads run along a
// row and the stores along the rows of a chunk, both coalesced.
template <typename RowFn>
__device__ __forceinline__ void image_slice(RowFn row, int n, int n_pad, int c0, int nc, uint4* __restrict__ dst,
                                            uint4 (*tile)[kImgSub + 1]) {
  for (int cs = 0; cs < nc; cs += kImgSub) {
    const int w = min(kImgSub, nc - cs);
    const int total = n_pad * kImgSub;
    uint4 v[kLtMaxN * kImgSub / 256];  // at most 4 per thread (256 threads)
#pragma unroll
    for (int u = 0; u < kLtMaxN * kImgSub / 256; ++u) {
      const int idx = threadIdx.x + u * blockDim.x, r = idx / kImgSub, cc = idx % kImgSub;
      v[u] = make_uint4(0, 0, 0, 0);
      if (idx < total && r < n && cc < w) v[u] = row(r)[c0 + cs + cc];
    }
#pragma unroll
    for (int u = 0; u < kLtMaxN * kImgSub / 256; ++u) {
      const int idx = threadIdx.x + u * blockDim.x;
      if (idx < total) tile[idx / kImgSub][idx % kImgSub] = bf16x8_to_f16x8(v[u]);
    }
    __syncthreads();
    for (int idx = threadIdx.x; idx < w * n_pad; idx += blockDim.x) {
      const int cc = idx / n_pad, r = idx - cc * n_pad;
      dst[(int64_t)(c0 + cs + cc) * n_pad + r] = tile[r][cc];
    }
    __syncthreads();
  }
}

// Block (tt, cs) writes column slice cs of plain token tile tt (x rows
// [64 tt, 64 tt + 64)) into the operand image; block (0, 0) also writes the
// plain token tiles, which the router and the shared expert use.
__global__ void lt_prep_kernel(const PrepParams P) {
  griddep_launch_dependents();
  griddep_wait();  // (the previous kernel in the stream wrote what this one reads, or reads what it writes)
  const int tt = blockIdx.x, cs = blockIdx.y;
  const int n = min(kLtMaxN, P.T - kLtMaxN * tt), n_pad = round16(n);
  if (tt == 0 && cs == 0) {
    for (int i = threadIdx.x; i < P.n_sh; i += blockDim.x) {
      const int ni = min(kLtMaxN, P.T - kLtMaxN * i);
      P.tiles[i] = LtTile{-1, P.T * P.k + kLtMaxN * i, ni, round16(ni), kLtMaxN * i, {0, 0, 0}};
    }
    if (threadIdx.x == 0) P.counters[6] = P.n_items1;
  }
  {
    const int nb = gridDim.x * gridDim.y, b = blockIdx.y * gridDim.x + blockIdx.x;
    for (int i = b * blockDim.x + threadIdx.x; i < P.n_bits; i += nb * blockDim.x) P.bits[i] = 0u;
  }
  __shared__ uint4 tile[kLtMaxN][kImgSub + 1];
  const int nc = P.H / 8 / kColSlices;
  const uint4* x4 = reinterpret_cast<const uint4*>(P.x);
  const int64_t rs = P.H / 8, r0 = (int64_t)kLtMaxN * tt;
  image_slice([&](int r) { return x4 + (r0 + r) * rs; }, n, n_pad, cs * nc, nc,
              reinterpret_cast<uint4*>(P.xg + r0 * P.H * 2), tile);
}

__device__ __forceinline__ bool topk_better(float v, int i, float bv, int bi) {
  return v > bv || (v == bv && i < bi);
}

// One warp per token.  NPER = experts per lane (lane l holds e = l + 32 i).
template <int NPER>
__global__ void lt_topk_kernel(const float* __restrict__ logits, const float* __restrict__ bias, int T, int E,
                               int E_pad, int k, int* __restrict__ ids, float* __restrict__ gates,
                               uint32_t* __restrict__ bits) {
  griddep_launch_dependents();
  griddep_wait();  // (the previous kernel in the stream wrote what this one reads, or reads what it writes)
  const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5), lane = threadIdx.x & 31;
  if (t >= T) return;
  const int64_t plane = (int64_t)T * E_pad;
  const float* l0 = logits + (int64_t)t * E_pad;
  float v[NPER];
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const int e = lane + 32 * i;
    float x = -INFINITY;
    if (e < E) {
      // the planes' logits, scaled back by 2^-11 and 2^-22 (exact)
      x = fmaf(l0[2 * plane + e], 0x1p-22f, fmaf(l0[plane + e], 0x1p-11f, l0[e])) + (bias ? bias[e] : 0.f);
      if (x != x) x = -INFINITY;
    }
    v[i] = x;
  }
  uint32_t taken = 0;
  float sel[kMaxTopK];
  int seli[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    if (j < k) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int i = 0; i < NPER; ++i) {
        const int e = lane + 32 * i;
        if (e < E && !((taken >> i) & 1u) && topk_better(v[i], e, bv, bi)) {
          bv = v[i];
          bi = e;
        }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (topk_better(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
      sel[j] = bv;
      seli[j] = bi;
    }
  }
  if (lane == 0) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) s += expf(sel[j] - sel[0]);
    const int W = (T + 31) / 32;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) {
        ids[t * k + j] = seli[j];
        gates[t * k + j] = expf(sel[j] - sel[0]) / s;
        atomicOr(&bits[(int64_t)seli[j] * W + (t >> 5)], 1u << (t & 31));  // token t chose expert seli[j]
      }
  }
}

struct PermParams {
  const int* ids;
  const uint32_t* bits;  // [E][ceil(T/32)]: bit t of expert e set when token t chose e
  int T, E, k, H, I, Ish, n_sh, prow_sh;
  int e0, n_e;  // routed experts held: token tiles only for [e0, e0 + n_e), by local index
  int* offsets;
  int* perm;
  int* pos;
  LtTile* tiles;
  int* counters;
};

constexpr int kPermWarps = 8;  // experts per block in lt_perm (one warp each)

// Pair p = t*k + j goes to slot offsets[e] + (number of tokens t' < t that
// chose e): expert e's tokens are the set bits of its bitmap row, so a
// pair's rank is the popcount of the bits below its token.  The k experts of
// one token are distinct, so the order of pairs within an expert is the
// order of their tokens.
//
// Every block reads all the rows' popcounts (one warp reduction per expert)
// and scans them, so it knows every expert's offset and tile position
// without waiting for another block; then warp w scatters expert
// blockIdx.x * kPermWarps + w and writes its token tiles.
__global__ void __launch_bounds__(kPermWarps * 32) lt_perm_kernel(const PermParams P) {
  griddep_launch_dependents();
  griddep_wait();  // (the previous kernel in the stream wrote what this one reads, or reads what it writes)
  __shared__ int off_s[kMaxE + 1];  // exclusive prefix of the counts over all experts
  __shared__ int tb_s[kMaxE];       // ... of the held experts' token tiles
  __shared__ int pb_s[kMaxE];       // ... of their operand rows
  __shared__ int wt[3][kPermWarps + 1];
  const int E = P.E, k = P.k, T = P.T, W = (T + 31) / 32;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // counts: warp w takes experts w, w + 8, ...; lane l the words l, l + 32, ...
  for (int ea = warp; ea < E; ea += 4 * kPermWarps) {
    int c[4] = {0, 0, 0, 0};
    for (int g = lane; g < W; g += 32) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int e = ea + q * kPermWarps;
        if (e < E) c[q] += __popc(P.bits[(int64_t)e * W + g]);
      }
    }
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e = ea + q * kPermWarps;
      const int n = __reduce_add_sync(0xffffffffu, c[q]);
      if (lane == 0 && e < E) off_s[e] = n;  // the count, for now
    }
  }
  __syncthreads();
  // exclusive scans of counts, tiles and rows over the experts: thread i
  // takes experts 4i .. 4i + 3 (E <= 1024 = 4 x 256)
  int cv[4], tv[4], rv[4], sc = 0, st = 0, sr = 0;
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const int e = 4 * tid + q;
    const int cnt = e < E ? off_s[e] : 0;
    const int M = e >= P.e0 && e < P.e0 + P.n_e ? cnt : 0;
    const int ntt = (M + kLtMaxN - 1) / kLtMaxN;
    cv[q] = cnt;
    tv[q] = ntt;
    rv[q] = M > 0 ? kLtMaxN * (ntt - 1) + round16(M - kLtMaxN * (ntt - 1)) : 0;
    sc += cv[q];
    st += tv[q];
    sr += rv[q];
  }
  int ic = sc, it = st, ir = sr;  // inclusive warp scans
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int yc = __shfl_up_sync(0xffffffffu, ic, o), yt = __shfl_up_sync(0xffffffffu, it, o),
              yr = __shfl_up_sync(0xffffffffu, ir, o);
    if (lane >= o) {
      ic += yc;
      it += yt;
      ir += yr;
    }
  }
  if (lane == 31) {
    wt[0][warp] = ic;
    wt[1][warp] = it;
    wt[2][warp] = ir;
  }
  __syncthreads();  // (every count is read above before any offset is written below)
  if (tid < 3) {
    int run = 0;
    for (int w = 0; w < kPermWarps; ++w) {
      const int v = wt[tid][w];
      wt[tid][w] = run;
      run += v;
    }
    wt[tid][kPermWarps] = run;
  }
  __syncthreads();
  {
    int bc = wt[0][warp] + ic - sc, bt = wt[1][warp] + it - st, br = wt[2][warp] + ir - sr;
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const int e = 4 * tid + q;
      if (e < E) {
        off_s[e] = bc;
        tb_s[e] = bt;
        pb_s[e] = br;
      }
      bc += cv[q];
      bt += tv[q];
      br += rv[q];
    }
    if (tid == 0) off_s[E] = wt[0][kPermWarps];
  }
  __syncthreads();
  const int e = blockIdx.x * kPermWarps + warp;
  if (e < E) {
    // scatter: lane l takes words l, l + 32, ... of the row; a word's bits
    // are ranked after the bits of the words before it
    const int base = off_s[e];
    int run = 0;
    for (int g0 = 0; g0 < W; g0 += 32) {
      const int g = g0 + lane;
      uint32_t word = g < W ? P.bits[(int64_t)e * W + g] : 0u;
      const int cw = __popc(word);
      int incl = cw;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += y;
      }
      int r = run + incl - cw;
      while (word) {
        const int t = g * 32 + __ffs(word) - 1;
        word &= word - 1u;
        int j = 0;
        for (int jj = 0; jj < k; ++jj)
          if (P.ids[t * k + jj] == e) j = jj;
        P.perm[base + r] = t * k + j;
        P.pos[t * k + j] = base + r;
        ++r;
      }
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) P.offsets[e] = base;
    // routed token tiles of a held expert, by local index
    if (e >= P.e0 && e < P.e0 + P.n_e) {
      const int M = off_s[e + 1] - base, ntt = (M + kLtMaxN - 1) / kLtMaxN;
      for (int i = lane; i < ntt; i += 32) {
        const int ni = min(kLtMaxN, M - kLtMaxN * i);
        P.tiles[P.n_sh + tb_s[e] + i] =
            LtTile{e - P.e0, base + kLtMaxN * i, ni, round16(ni), P.prow_sh + pb_s[e] + kLtMaxN * i, {0, 0, 0}};
      }
    }
  }
  if (blockIdx.x == 0 && tid == 0) {
    const int n_tiles = wt[1][kPermWarps];
    const int n_gu = P.I / 64, n_dn = P.H / 128;
    P.offsets[E] = off_s[E];
    P.counters[7] = n_tiles * n_gu;                                   // routed gate/up items
    P.counters[8] = (P.Ish > 0 ? P.n_sh : 0) * n_dn + n_tiles * n_dn;  // down items
    P.counters[9] = n_tiles;
  }
}

// Block (b, cs) gathers column slice cs of routed tile n_sh + b (if it exists)
// into the operand image.
__global__ void lt_gather_kernel(const __nv_bfloat16* __restrict__ x, const int* __restrict__ perm,
                                 const LtTile* __restrict__ tiles, const int* __restrict__ counters, int n_sh, int k,
                                 int H, uint8_t* __restrict__ xg) {
  griddep_launch_dependents();
  griddep_wait();  // (the previous kernel in the stream wrote what this one reads, or reads what it writes)
  if ((int)blockIdx.x >= counters[9]) return;
  const LtTile tl = tiles[n_sh + blockIdx.x];
  __shared__ int tok[kLtMaxN];
  for (int r = threadIdx.x; r < tl.n; r += blockDim.x) tok[r] = perm[tl.slot0 + r] / k;
  __syncthreads();
  __shared__ uint4 tile[kLtMaxN][kImgSub + 1];
  const int nc = H / 8 / kColSlices;
  const uint4* x4 = reinterpret_cast<const uint4*>(x);
  const int64_t rs = H / 8;
  image_slice([&](int r) { return x4 + (int64_t)tok[r] * rs; }, tl.n, tl.n_pad, blockIdx.y * nc, nc,
              reinterpret_cast<uint4*>(xg + (int64_t)tl.prow0 * H * 2), tile);
}

// y[t] = sum_j g[t,j] z[pos[t,j]] + z[T k + t]; one block per token, 8 columns per thread step.
// Pairs whose expert the layer does not hold (an expert-parallel shard) are
// left out of the sum.
__global__ void __launch_bounds__(256, 4) lt_combine_kernel(const __nv_bfloat16* __restrict__ z, const float* __restrict__ gates,
                                  const int* __restrict__ pos, const int* __restrict__ ids, int e0, int n_e, int T,
                                  int k, int H, bool shared, const __nv_bfloat16* __restrict__ xres,
                                  __nv_bfloat16* __restrict__ y) {
  griddep_launch_dependents();
  griddep_wait();  // (the previous kernel in the stream wrote what this one reads, or reads what it writes)
  const int t = blockIdx.x;
  __shared__ float g[kMaxTopK];
  __shared__ int ps[kMaxTopK];
  __shared__ int nk;
  if (threadIdx.x == 0) {
    // the held pairs, in slot order
    int n = 0;
    for (int j = 0; j < k; ++j) {
      const int e = ids[t * k + j];
      if (e >= e0 && e < e0 + n_e) {
        g[n] = gates[t * k + j];
        ps[n] = pos[t * k + j];
        ++n;
      }
    }
    nk = n;
  }
  __syncthreads();
  const int kh = nk;
  for (int c = threadIdx.x; c < H / 8; c += blockDim.x) {
    float acc[8];
#pragma unroll
    for (int m = 0; m < 8; ++m) acc[m] = 0.f;
    // the slots' loads in flight 8 at a time, then their sums (in slot order)
    for (int j0 = 0; j0 < kh; j0 += 8) {
      uint4 zu[8];
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j0 + j < kh) zu[j] = *reinterpret_cast<const uint4*>(z + (int64_t)ps[j0 + j] * H + 8 * c);
#pragma unroll
      for (int j = 0; j < 8; ++j)
        if (j0 + j < kh) {
          const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&zu[j]);
#pragma unroll
          for (int m = 0; m < 8; ++m) acc[m] += g[j0 + j] * __bfloat162float(b[m]);
        }
    }
    if (shared) {
      const uint4 u = *reinterpret_cast<const uint4*>(z + (int64_t)(T * k + t) * H + 8 * c);
      const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
      for (int m = 0; m < 8; ++m) acc[m] += __bfloat162float(b[m]);
    }
    if (xres) {
      const uint4 u = *reinterpret_cast<const uint4*>(xres + (int64_t)t * H + 8 * c);
      const __nv_bfloat16* b = reinterpret_cast<const __nv_bfloat16*>(&u);
#pragma unroll
      for (int m = 0; m < 8; ++m) acc[m] += __bfloat162float(b[m]);
    }
    uint4 o;
    uint32_t* ow = reinterpret_cast<uint32_t*>(&o);
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      const __nv_bfloat162 v = __floats2bfloat162_rn(acc[2 * m], acc[2 * m + 1]);
      ow[m] = *reinterpret_cast<const uint32_t*>(&v);
    }
    *reinterpret_cast<uint4*>(y + (int64_t)t * H + 8 * c) = o;
  }
}

size_t align256(size_t v) { return (v + 255) / 256 * 256; }

#define LT_CK(call)                       \
  do {                                    \
    cudaError_t e_ = (call);              \
    if (e_ != cudaSuccess) return e_;     \
  } while (0)

}  // namespace

// ---------------------------------------------------------------------------
// Host side
// ---------------------------------------------------------------------------

bool large_t_enabled(const moe_layer* L) { return L->T_max > kMaxSmallT; }

// Allocates the LT weight copies and the workspace.  Shapes were validated by
// the caller (H % 128 == 0, I and I_shared multiples of 64).
cudaError_t large_t_alloc(moe_layer* L) {
  LtState* S = new LtState();
  L->lt = S;
  const int H = L->H, E = L->E, I = L->I, Ish = L->Ish, k = L->k, Tm = L->T_max;
  S->E_pad128 = (E + 127) / 128 * 128;
  S->Imax = std::max(I, Ish);
  S->gu_stride = (int64_t)(I / 64) * lt_tile_bytes(L->fmt, H);
  S->dn_stride = (int64_t)(H / 128) * lt_tile_bytes(L->fmt, I);
  S->router_plane = (int64_t)(S->E_pad128 / 128) * lt_tile_bytes(MOE_BF16, H);
  LT_CK(cudaMalloc(&S->gu, (size_t)S->gu_stride * L->n_e));
  LT_CK(cudaMalloc(&S->dn, (size_t)S->dn_stride * L->n_e));
  LT_CK(cudaMalloc(&S->router, (size_t)S->router_plane * kLtPlanes));
  size_t wb = (size_t)(S->gu_stride + S->dn_stride) * L->n_e + (size_t)S->router_plane * kLtPlanes;
  if (Ish > 0) {
    const size_t a = (size_t)(Ish / 64) * lt_tile_bytes(L->sfmt, H), b = (size_t)(H / 128) * lt_tile_bytes(L->sfmt, Ish);
    LT_CK(cudaMalloc(&S->sgu, a));
    LT_CK(cudaMalloc(&S->sdn, b));
    wb += a + b;
  }
  S->weight_bytes = wb;

  const int n_sh_max = (Tm + kLtMaxN - 1) / kLtMaxN;
  const int Tk = Tm * k;
  // routed tiles: sum over experts of ceil(M_e / 64) <= T k / 64 + min(E, T k)
  S->max_tiles = n_sh_max + std::min(E, Tk) + Tk / kLtMaxN + 1;
  S->max_rows = Tm + Tk + 16 * S->max_tiles;
  size_t off = 0;
  auto take = [&](size_t b) {
    const size_t o = off;
    off = align256(off + b);
    return o;
  };
  const size_t o_cnt = take(16 * 4);
  const size_t o_status = take(16);
  const size_t o_logits = take((size_t)kLtPlanes * Tm * S->E_pad128 * 4);
  const size_t o_ids = take((size_t)Tk * 4);
  const size_t o_bits = take((size_t)E * ((Tm + 31) / 32) * 4);
  const size_t o_gates = take((size_t)Tk * 4);
  const size_t o_pos = take((size_t)Tk * 4);
  const size_t o_perm = take((size_t)Tk * 4);
  const size_t o_offs = take((size_t)(E + 1) * 4);
  const size_t o_tiles = take((size_t)S->max_tiles * sizeof(LtTile));
  const size_t o_xg = take((size_t)S->max_rows * H * 2);
  const size_t o_h = take((size_t)S->max_rows * S->Imax * 2);
  const size_t o_z = take((size_t)(Tk + Tm) * H * 2);
  S->ws_bytes = off;
  LT_CK(cudaMalloc(&S->ws, S->ws_bytes));
  LT_CK(cudaMemset(S->ws, 0, o_status + 16));
  uint8_t* w = static_cast<uint8_t*>(S->ws);
  S->counters = reinterpret_cast<int*>(w + o_cnt);
  S->status = reinterpret_cast<int*>(w + o_status);
  S->logits = reinterpret_cast<float*>(w + o_logits);
  S->ids = reinterpret_cast<int*>(w + o_ids);
  S->bits = reinterpret_cast<uint32_t*>(w + o_bits);
  S->gates = reinterpret_cast<float*>(w + o_gates);
  S->pos = reinterpret_cast<int*>(w + o_pos);
  S->perm = reinterpret_cast<int*>(w + o_perm);
  S->offsets = reinterpret_cast<int*>(w + o_offs);
  S->tiles = reinterpret_cast<LtTile*>(w + o_tiles);
  S->xg = w + o_xg;
  S->h = w + o_h;
  S->z = reinterpret_cast<__nv_bfloat16*>(w + o_z);
  LT_CK(lt_gemm_configure());
  return cudaSuccess;
}

// which: 0 gate, 1 up, 2 down, 3 shared gate, 4 shared up, 5 shared down.
cudaError_t large_t_repack(moe_layer* L, int which, int e, const uint8_t* src, cudaStream_t st) {
  LtState* S = L->lt;
  const bool sh = which >= 3;
  const int fmt = sh ? L->sfmt : L->fmt;
  const int kind = which % 3;
  const int I = sh ? L->Ish : L->I;
  const int rows = kind == 2 ? L->H : I, K = kind == 2 ? I : L->H;
  uint8_t* dst = kind == 2 ? (sh ? S->sdn : S->dn + (int64_t)e * S->dn_stride)
                           : (sh ? S->sgu : S->gu + (int64_t)e * S->gu_stride);
  const int mode = kind == 2 ? 0 : (kind == 0 ? 1 : 2);
  const int64_t n = (int64_t)rows * (fmt == MOE_Q8_0 ? K / 32 : K / 256);
  const unsigned grid = (unsigned)((n + 255) / 256);
  if (fmt == MOE_Q8_0)
    lt_repack_q8_kernel<<<grid, 256, 0, st>>>(src, dst, rows, K, mode);
  else
    lt_repack_q4ks_kernel<<<grid, 256, 0, st>>>(src, dst, rows, K, mode);
  return cudaGetLastError();
}

cudaError_t large_t_repack_router(moe_layer* L, const float* src, cudaStream_t st) {
  LtState* S = L->lt;
  const int64_t n = (int64_t)S->E_pad128 * (L->H / 8);
  lt_repack_router_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(src, S->router, L->E, S->E_pad128, L->H,
                                                                       S->router_plane);
  return cudaGetLastError();
}

size_t large_t_weight_bytes(const moe_layer* L) { return L->lt ? L->lt->weight_bytes : 0; }
size_t large_t_workspace_bytes(const moe_layer* L) { return L->lt ? L->lt->ws_bytes : 0; }
int* large_t_status_word(const moe_layer* L) { return L->lt ? L->lt->status : nullptr; }
int* large_t_counters(const moe_layer* L) { return L->lt ? L->lt->counters : nullptr; }

cudaError_t large_t_forward(moe_layer* L, const void* x, int T, void* y, bool residual, cudaStream_t st) {
  LtState* S = L->lt;
  const int H = L->H, E = L->E, k = L->k;
  const int n_sh = (T + kLtMaxN - 1) / kLtMaxN;
  const int prow_sh = kLtMaxN * (n_sh - 1) + round16(T - kLtMaxN * (n_sh - 1));
  const int n_rt_r = S->E_pad128 / 128;
  const int n_rt_items = kLtPlanes * n_rt_r * n_sh;
  const int n_gu_sh = L->Ish / 64;

  PrepParams pp{static_cast<const __nv_bfloat16*>(x), T, H, k, n_sh, n_rt_items + n_gu_sh * n_sh, S->tiles,
                S->counters, S->xg, S->bits, E * ((T + 31) / 32)};
  LT_CK(launch_pdl(lt_prep_kernel, dim3(n_sh, kColSlices), 256, 0, st, pp));

  LtGemmParams g{};
  g.tiles = S->tiles;
  g.status = S->status;
  g.gu = S->gu; g.dn = S->dn; g.sgu = S->sgu; g.sdn = S->sdn; g.router = S->router;
  g.gu_stride = S->gu_stride; g.dn_stride = S->dn_stride; g.router_plane = S->router_plane;
  g.fmt = L->fmt; g.sfmt = L->sfmt;
  g.H = H; g.I = L->I; g.Ish = L->Ish; g.Imax = S->Imax; g.E_pad128 = S->E_pad128; g.T = T; g.k = k;
  g.xg = S->xg; g.h = S->h; g.z = S->z; g.logits = S->logits;
  g.timeout_ns = L->timeout_ns;
  g.n_rt_router = n_rt_r;
  g.n_router_tiles = n_sh;
  const int grid = L->num_sms;

  // router logits + shared-expert gate/up (plain token tiles)
  g.n_items = S->counters + 6; g.queue = S->counters + 0; g.exit_cnt = S->counters + 3;
  g.n_rt_items = n_rt_items; g.tile_kind = kItemGU; g.tile0 = 0; g.n_rt_tile = n_gu_sh > 0 ? n_gu_sh : 1;
  LT_CK(lt_gemm_launch(g, grid, st));

  const int warps = 8;
  const unsigned tgrid = (unsigned)((T + warps - 1) / warps);
  const int nper = (E + 31) / 32;
#define LT_TOPK(NP)                                                                                               \
  launch_pdl(lt_topk_kernel<NP>, tgrid, warps * 32, 0, st, (const float*)S->logits, (const float*)L->router_b, T, E, \
             S->E_pad128, k, S->ids, S->gates, S->bits)
  if (nper <= 4) LT_CK(LT_TOPK(4));
  else if (nper <= 8) LT_CK(LT_TOPK(8));
  else if (nper <= 12) LT_CK(LT_TOPK(12));
  else if (nper <= 16) LT_CK(LT_TOPK(16));
  else LT_CK(LT_TOPK(32));
#undef LT_TOPK

  PermParams P{S->ids, S->bits, T, E, k, H, L->I, L->Ish, n_sh, prow_sh, L->e0, L->n_e, S->offsets, S->perm, S->pos,
               S->tiles, S->counters};
  LT_CK(launch_pdl(lt_perm_kernel, (E + kPermWarps - 1) / kPermWarps, kPermWarps * 32, 0, st, P));

  const int max_routed = S->max_tiles - (L->T_max + kLtMaxN - 1) / kLtMaxN;
  LT_CK(launch_pdl(lt_gather_kernel, dim3(max_routed, kColSlices), 256, 0, st, static_cast<const __nv_bfloat16*>(x),
                   (const int*)S->perm, (const LtTile*)S->tiles, (const int*)S->counters, n_sh, k, H, S->xg));

  // routed gate/up
  g.n_items = S->counters + 7; g.queue = S->counters + 1; g.exit_cnt = S->counters + 4;
  g.n_rt_items = 0; g.tile_kind = kItemGU; g.tile0 = n_sh; g.n_rt_tile = L->I / 64;
  LT_CK(lt_gemm_launch(g, grid, st));
  // down projections: shared tiles (if any) then routed tiles
  g.n_items = S->counters + 8; g.queue = S->counters + 2; g.exit_cnt = S->counters + 5;
  g.n_rt_items = 0; g.tile_kind = kItemDN; g.tile0 = L->Ish > 0 ? 0 : n_sh; g.n_rt_tile = H / 128;
  LT_CK(lt_gemm_launch(g, grid, st));

  LT_CK(launch_pdl(lt_combine_kernel, T, 256, 0, st, (const __nv_bfloat16*)S->z, (const float*)S->gates,
                   (const int*)S->pos, (const int*)S->ids, L->e0, L->n_e, T, k, H, L->Ish > 0,
                   residual ? static_cast<const __nv_bfloat16*>(x) : nullptr, static_cast<__nv_bfloat16*>(y)));
  return cudaSuccess;
}

cudaError_t large_t_get_routing(moe_layer* L, int32_t* ids, float* gates, int32_t* offsets, int32_t* perm,
                                cudaStream_t st) {
  LtState* S = L->lt;
  const size_t Tk = (size_t)L->last_T * L->k;
  if (ids) LT_CK(cudaMemcpyAsync(ids, S->ids, Tk * 4, cudaMemcpyDeviceToDevice, st));
  if (gates) LT_CK(cudaMemcpyAsync(gates, S->gates, Tk * 4, cudaMemcpyDeviceToDevice, st));
  if (offsets) LT_CK(cudaMemcpyAsync(offsets, S->offsets, (size_t)(L->E + 1) * 4, cudaMemcpyDeviceToDevice, st));
  if (perm) LT_CK(cudaMemcpyAsync(perm, S->perm, Tk * 4, cudaMemcpyDeviceToDevice, st));
  return cudaSuccess;
}

void large_t_release(moe_layer* L) {
  LtState* S = L->lt;
  if (!S) return;
  cudaFree(S->gu);
  cudaFree(S->dn);
  cudaFree(S->sgu);
  cudaFree(S->sdn);
  cudaFree(S->router);
  cudaFree(S->ws);
  delete S;
  L->lt = nullptr;
}

}  // namespace moe
