// mtp.cu -- the output head entry points and one MTP draft/verify round.
//
// mtp_round sequences, on the caller's stream: the pre-norm residual target
// blocks (one launch each: the layer adds its output to h and normalises the
// next block's input), the output norm + LM head on the verify batch, the
// noisy draft rows,
// the draft heads, the LM head on the draft rows, their argmax, and greedy
// acceptance.  Everything runs in this library's kernels; nothing allocates.
// The residual stream (the hidden state h between blocks, and the noisy draft
// rows) is kept in fp32 whatever the activation type; only the inputs and
// outputs of the MoE layers are in the act dtype (as in the pages' runtime,
// whose hidden states between operations are F32 tensors).
#include <utility>

#include "layer.cuh"

namespace moe {
cudaError_t lm_repack(const uint8_t* src, uint8_t* dst, int V, int H, cudaStream_t st);
cudaError_t lm_configure(int H, int max_optin);
Chunking lm_chunking(int H);
size_t lm_weight_bytes(int V, int H, Chunking ch);
cudaError_t lm_forward(const moe_lm_head* lm, const void* x, bool x_f32, int T, float eps, float* logits,
                       cudaStream_t st);
size_t accept_workspace_bytes(int k, int V);
cudaError_t accept_launch_cut(int32_t* draft, int k, const float* logits, int V, const float* dprob, float p_min,
                              int32_t* out_n, int32_t* out_next, void* ws, cudaStream_t st);

namespace {

template <int L>
__device__ __forceinline__ float ld_act(const void* p, int64_t i) {
  if constexpr (L == 2) return __bfloat162float(static_cast<const __nv_bfloat16*>(p)[i]);
  else return static_cast<const float*>(p)[i];
}
template <int L>
__device__ __forceinline__ float st_act(void* p, int64_t i, float v) {  // returns the stored value
  if constexpr (L == 2) {
    const __nv_bfloat16 b = __float2bfloat16_rn(v);
    static_cast<__nv_bfloat16*>(p)[i] = b;
    return __bfloat162float(b);
  } else {
    static_cast<float*>(p)[i] = v;
    return v;
  }
}

// Sum over the block (blockDim.x == 256).
__device__ __forceinline__ float block_sum(float v, float* red) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  float s = 0.f;
  for (int w = 0; w < 8; ++w) s += red[w];
  __syncthreads();
  return s;
}

// One row per block: h_out = h_in + y (fp32; y is the layer's fp32 output;
// without y, h_out = h_in) and xn = rmsnorm(h_out) (act dtype).  h_in is fp32
// (LIN = 4) or the act dtype (LIN = L: the round's input batch).
template <int L, int LIN>
__global__ void __launch_bounds__(256) add_rmsnorm_kernel(const void* __restrict__ h_in, const float* __restrict__ y,
                                                          float* __restrict__ h_out, void* __restrict__ xn, int H,
                                                          float eps) {
  __shared__ float red[8];
  griddep_launch_dependents();
  griddep_wait();
  const int64_t base = (int64_t)blockIdx.x * H;
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    float v = ld_act<LIN>(h_in, base + c);
    if (y) v += y[base + c];
    h_out[base + c] = v;
    ss = fmaf(v, v, ss);
  }
  __syncthreads();  // h_out written by this block before it is read back
  const float inv = 1.f / sqrtf(block_sum(ss, red) / (float)H + eps);
  for (int c = threadIdx.x; c < H; c += blockDim.x) st_act<L>(xn, base + c, h_out[base + c] * inv);
}

// Block (j, i), i <= j: v = h[i] + noise[j][i] (fp32); hin[j][i] =
// rmsnorm(v) (the head's input, act dtype) and, for i == j, rows[j] = v
// (fp32: the row the draft is read from).
template <int L>
__global__ void __launch_bounds__(256) draft_rows_kernel(const float* __restrict__ h, const float* __restrict__ noise,
                                                         int k, int H, float eps, void* __restrict__ hin,
                                                         float* __restrict__ rows) {
  __shared__ float red[8];
  griddep_launch_dependents();
  griddep_wait();
  const int j = blockIdx.x / k, i = blockIdx.x % k;
  if (i > j) return;
  const int64_t src = (int64_t)i * H, nz = ((int64_t)j * k + i) * H;
  float ss = 0.f;
  for (int c = threadIdx.x; c < H; c += blockDim.x) {
    const float v = h[src + c] + noise[nz + c];
    ss = fmaf(v, v, ss);
    if (i == j) rows[(int64_t)j * H + c] = v;
  }
  const float inv = 1.f / sqrtf(block_sum(ss, red) / (float)H + eps);
  for (int c = threadIdx.x; c < H; c += blockDim.x) st_act<L>(hin, nz + c, (h[src + c] + noise[nz + c]) * inv);
}

// ids[r] = argmax of row r (lowest index on ties) and probs[r] = the softmax
// probability of that token, 1 / sum_v exp(l_v - max l) (the draft's
// confidence, for the --spec-draft-p-min cut); one CTA of kArgThreads per
// row.  With V % 4 == 0 each thread reads float4 c4 = t, t + kArgThreads, ...
// eight loads at a time, all in flight before the compares.  The sum is an
// online one: each thread keeps sum exp(v - m) for its running maximum m and
// rescales it when m grows; partial sums merge as s1 e^(m1 - m) + s2 e^(m2 - m)
// in a fixed order, so the result is deterministic.
constexpr int kArgThreads = 1024;

__device__ __forceinline__ void merge_sum(float& m, float& s, float om, float os) {
  if (om == -INFINITY) return;
  if (m == -INFINITY) {
    m = om;
    s = os;
    return;
  }
  const float nm = fmaxf(m, om);
  s = s * expf(m - nm) + os * expf(om - nm);
  m = nm;
}

__global__ void __launch_bounds__(kArgThreads) argmax_rows_kernel(const float* __restrict__ logits, int V,
                                                                  int32_t* __restrict__ ids,
                                                                  float* __restrict__ probs) {
  __shared__ float sv[kArgThreads / 32];
  __shared__ int si[kArgThreads / 32];
  __shared__ float ss[kArgThreads / 32];
  griddep_launch_dependents();
  griddep_wait();
  const float* row = logits + (int64_t)blockIdx.x * V;
  float bv = -INFINITY;
  int bi = 0x7fffffff;
  float sum = 0.f;  // sum of exp(v - bv) over the values seen
  // per thread the indices visited increase, so strict > keeps the lowest
  auto take = [&](float v, int c) {
    if (v > bv || bi == 0x7fffffff) {
      sum = bi == 0x7fffffff ? 1.f : fmaf(sum, expf(bv - v), 1.f);
      bv = v;
      bi = c;
    } else {
      sum += expf(v - bv);
    }
  };
  if ((V & 3) == 0) {
    const float4* r4 = reinterpret_cast<const float4*>(row);
    const int n4 = V / 4;
    for (int c0 = threadIdx.x; c0 < n4; c0 += 8 * kArgThreads) {
      float4 a[8];
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c0 + u * kArgThreads < n4) a[u] = __ldg(r4 + c0 + u * kArgThreads);
#pragma unroll
      for (int u = 0; u < 8; ++u)
        if (c0 + u * kArgThreads < n4) {
          const int c = 4 * (c0 + u * kArgThreads);
          take(a[u].x, c);
          take(a[u].y, c + 1);
          take(a[u].z, c + 2);
          take(a[u].w, c + 3);
        }
    }
  } else {
    for (int c = threadIdx.x; c < V; c += kArgThreads) take(row[c], c);
  }
  float sm = bi == 0x7fffffff ? -INFINITY : bv;  // the maximum the sum refers to
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    const float ov = __shfl_xor_sync(0xffffffffu, bv, o);
    const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
    const float om = __shfl_xor_sync(0xffffffffu, sm, o);
    const float os = __shfl_xor_sync(0xffffffffu, sum, o);
    if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    merge_sum(sm, sum, om, os);
  }
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (lane == 0) { sv[warp] = bv; si[warp] = bi; ss[warp] = sum; }
  __syncthreads();
  if (threadIdx.x == 0) {
    sm = sv[0];
    for (int w = 1; w < kArgThreads / 32; ++w) {
      merge_sum(sm, sum, sv[w], ss[w]);
      if (sv[w] > bv || (sv[w] == bv && si[w] < bi)) { bv = sv[w]; bi = si[w]; }
    }
    ids[blockIdx.x] = bi;
    if (probs) probs[blockIdx.x] = 1.f / sum;
  }
}

size_t al256(size_t v) { return (v + 255) / 256 * 256; }

struct RoundLayout {
  size_t hA, hB, xn, xn2, hin, hout, rows, dlog, dprob, acc, total;
};
RoundLayout round_layout(int H, int k, int V, int act) {
  const size_t esz = act == MOE_ACT_BF16 ? 2 : 4;
  RoundLayout r{};
  size_t off = 0;
  auto take = [&](size_t b) { const size_t o = off; off = al256(off + b); return o; };
  r.acc = take(accept_workspace_bytes(k, V));  // must stay zero between calls: first
  r.hA = take((size_t)(k + 1) * H * 4);  // residual stream: fp32
  r.hB = take((size_t)(k + 1) * H * 4);
  r.xn = take((size_t)(k + 1) * H * esz);
  r.xn2 = take((size_t)(k + 1) * H * esz);  // the normalised rows ping-pong with xn
  r.hin = take((size_t)k * k * H * esz);
  r.hout = take((size_t)k * k * H * esz);
  r.rows = take((size_t)k * H * 4);
  r.dlog = take((size_t)k * V * 4);
  r.dprob = take((size_t)k * 4);
  r.total = off;
  return r;
}

}  // namespace
}  // namespace moe

using namespace moe;

#define MCK(call, what)                                                                      \
  do {                                                                                       \
    cudaError_t e_ = (call);                                                                 \
    if (e_ != cudaSuccess) return set_error(MOE_ECUDA, "%s: %s", what, cudaGetErrorString(e_)); \
  } while (0)

extern "C" {

int moe_lm_head_create(const moe_tensor* w, int32_t T_max, int32_t act_dtype, void* stream, moe_lm_head** out) {
  if (!w || !out) return set_error(MOE_EINVAL, "moe_lm_head_create: NULL argument");
  if (w->fmt != MOE_Q8_0) return set_error(MOE_EFORMAT, "moe_lm_head_create: the output matrix must be Q8_0");
  if (w->reserved != 0) return set_error(MOE_EINVAL, "moe_lm_head_create: reserved field must be 0");
  const int64_t V = w->rows, H = w->cols;
  if (V < 1 || V > (1 << 24) || H <= 0 || H % 512 || H > 16384)
    return set_error(MOE_EINVAL, "moe_lm_head_create: shape [V, H] must have 1 <= V <= 2^24, H a multiple of 512 <= 16384");
  if (T_max < 1 || T_max > 8) return set_error(MOE_EINVAL, "moe_lm_head_create: T_max outside 1..8");
  if (act_dtype != MOE_ACT_BF16 && act_dtype != MOE_ACT_F32) return set_error(MOE_EINVAL, "moe_lm_head_create: act_dtype");
  if (!w->data || w->nbytes != (size_t)V * (H / 32) * 34)
    return set_error(MOE_EINVAL, "moe_lm_head_create: data NULL or nbytes != V * H / 32 * 34");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  moe_lm_head* lm = new moe_lm_head();
  lm->V = (int)V;
  lm->H = (int)H;
  lm->T_max = T_max;
  lm->act = act_dtype;
  uint8_t* staged = nullptr;
  auto cleanup = [&](int rc) {
    if (staged) cudaFree(staged);
    if (rc != MOE_OK) moe_lm_head_destroy(lm);
    return rc;
  };
  cudaError_t e;
  if ((e = cudaGetDevice(&lm->dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&lm->num_sms, cudaDevAttrMultiProcessorCount, lm->dev)) != cudaSuccess ||
      (e = cudaDeviceGetAttribute(&lm->max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, lm->dev)) != cudaSuccess)
    return cleanup(set_error(MOE_ECUDA, "%s", cudaGetErrorString(e)));
  if ((e = cudaMalloc(&lm->w, lm_weight_bytes((int)V, (int)H, lm_chunking((int)H)))) != cudaSuccess ||
      (e = cudaMalloc(&lm->status, 16)) != cudaSuccess || (e = cudaMemsetAsync(lm->status, 0, 16, st)) != cudaSuccess)
    return cleanup(set_error(e == cudaErrorMemoryAllocation ? MOE_ENOMEM : MOE_ECUDA, "%s", cudaGetErrorString(e)));
  cudaPointerAttributes pa{};
  const uint8_t* src = static_cast<const uint8_t*>(w->data);
  if (cudaPointerGetAttributes(&pa, w->data) != cudaSuccess || pa.type != cudaMemoryTypeDevice) {
    cudaGetLastError();
    if ((e = cudaMalloc(&staged, w->nbytes)) != cudaSuccess ||
        (e = cudaMemcpyAsync(staged, w->data, w->nbytes, cudaMemcpyHostToDevice, st)) != cudaSuccess)
      return cleanup(set_error(e == cudaErrorMemoryAllocation ? MOE_ENOMEM : MOE_ECUDA, "%s", cudaGetErrorString(e)));
    src = staged;
  }
  if ((e = lm_repack(src, lm->w, (int)V, (int)H, st)) != cudaSuccess || (e = lm_configure((int)H, lm->max_optin)) != cudaSuccess ||
      (e = cudaStreamSynchronize(st)) != cudaSuccess)
    return cleanup(set_error(MOE_ECUDA, "%s", cudaGetErrorString(e)));
  *out = lm;
  return cleanup(MOE_OK);
}

int moe_lm_head_forward(moe_lm_head* lm, const void* x, int32_t T, float eps, float* logits, void* stream) {
  if (!lm) return set_error(MOE_EINVAL, "moe_lm_head_forward: NULL head");
  if (T < 0 || T > lm->T_max) return set_error(MOE_EINVAL, "moe_lm_head_forward: T outside 0..T_max");
  if (T == 0) return MOE_OK;
  if (!x || !logits) return set_error(MOE_EINVAL, "moe_lm_head_forward: NULL x or logits");
  if (reinterpret_cast<uintptr_t>(x) & 15) return set_error(MOE_EINVAL, "moe_lm_head_forward: x must be 16-byte aligned");
  if (!(eps >= 0.f)) return set_error(MOE_EINVAL, "moe_lm_head_forward: eps must be >= 0");
  cudaError_t e = lm_forward(lm, x, lm->act == MOE_ACT_F32, T, eps, logits, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return set_error(MOE_ECUDA, "moe_lm_head_forward: %s", cudaGetErrorString(e));
  return MOE_OK;
}

int moe_lm_head_status(moe_lm_head* lm, void* stream) {
  if (!lm) return set_error(MOE_EINVAL, "moe_lm_head_status: NULL head");
  cudaError_t e = cudaStreamSynchronize(static_cast<cudaStream_t>(stream));
  int word[4] = {0, 0, 0, 0};
  if (e == cudaSuccess) e = cudaMemcpy(word, lm->status, 16, cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return set_error(MOE_ECUDA, "moe_lm_head_status: %s", cudaGetErrorString(e));
  if (word[0] != 0) {
    e = cudaMemset(lm->status, 0, 16);
    if (e != cudaSuccess) return set_error(MOE_ECUDA, "moe_lm_head_status: %s", cudaGetErrorString(e));
    static const char* sites[] = {"?", "free stage", "full stage", "copy drain"};
    return set_error(MOE_ETIMEOUT, "a device-side wait of the LM head timed out: %s",
                     sites[(word[1] >= 0 && word[1] <= 3) ? word[1] : 0]);
  }
  return MOE_OK;
}

void moe_lm_head_destroy(moe_lm_head* lm) {
  if (!lm) return;
  cudaFree(lm->w);
  cudaFree(lm->status);
  delete lm;
}

size_t mtp_round_workspace_bytes(int32_t H, int32_t k, int32_t V, int32_t act_dtype) {
  if (H <= 0 || k < 1 || k > 7 || V < 1 || V > (1 << 24) || (act_dtype != MOE_ACT_BF16 && act_dtype != MOE_ACT_F32))
    return 0;
  return round_layout(H, k, V, act_dtype).total;
}

int mtp_round(moe_layer* const* target_layers, int32_t n_target, moe_layer* const* draft_heads, int32_t k,
              moe_lm_head* lm, const void* x, const float* noise, float eps, float p_min, void* workspace,
              size_t workspace_bytes, float* target_logits, float* draft_logits, void* head_out, int32_t* draft_ids,
              int32_t* out_n_accepted, int32_t* out_next_token, void* stream) {
  if (k < 1 || k > 7) return set_error(MOE_EINVAL, "mtp_round: k outside 1..7");
  if (n_target < 0 || (n_target > 0 && !target_layers) || !draft_heads || !lm || !x || !noise || !workspace ||
      !target_logits || !draft_ids || !out_n_accepted || !out_next_token)
    return set_error(MOE_EINVAL, "mtp_round: NULL argument");
  if (!(p_min >= 0.f)) return set_error(MOE_EINVAL, "mtp_round: p_min must be >= 0 (0 keeps every draft)");
  const int H = lm->H, act = lm->act, V = lm->V;
  if (lm->T_max < k + 1) return set_error(MOE_EINVAL, "mtp_round: the LM head's T_max is below k+1");
  for (int l = 0; l < n_target; ++l) {
    const moe_layer* L = target_layers[l];
    if (!L || L->H != H || L->act != act || L->T_max < k + 1)
      return set_error(MOE_EINVAL, "mtp_round: target layer %d: NULL, or H / act_dtype / T_max mismatch", l);
  }
  for (int j = 0; j < k; ++j) {
    const moe_layer* L = draft_heads[j];
    if (!L || L->H != H || L->act != act || L->T_max < j + 1)
      return set_error(MOE_EINVAL, "mtp_round: draft head %d: NULL, or H / act_dtype / T_max mismatch", j);
  }
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(head_out)) & 15)
    return set_error(MOE_EINVAL, "mtp_round: x and head_out must be 16-byte aligned");
  if (reinterpret_cast<uintptr_t>(workspace) & 255) return set_error(MOE_EINVAL, "mtp_round: workspace must be 256-byte aligned");
  const RoundLayout r = round_layout(H, k, V, act);
  if (workspace_bytes < r.total) return set_error(MOE_EINVAL, "mtp_round: workspace %zu bytes, need %zu", workspace_bytes, r.total);
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  const size_t esz = act == MOE_ACT_BF16 ? 2 : 4;
  int rc;
  cudaError_t e = cudaSuccess;
  // target stack: pre-norm residual blocks h <- h + MoE(rmsnorm(h)); the
  // hidden state ping-pongs between hA and hB, xn holds the normalised rows
  void* xn = w + r.xn;
  float* hA = reinterpret_cast<float*>(w + r.hA);
  float* hB = reinterpret_cast<float*>(w + r.hB);
  // h_0 = x (to fp32), xn = rmsnorm(h_0)
  if (act == MOE_ACT_BF16)
    e = launch_pdl(add_rmsnorm_kernel<2, 2>, k + 1, 256, 0, st, x, (const float*)nullptr, hA, xn, H, eps);
  else
    e = launch_pdl(add_rmsnorm_kernel<4, 4>, k + 1, 256, 0, st, x, (const float*)nullptr, hA, xn, H, eps);
  MCK(e, "mtp_round: norm");
  // each layer adds its output to h in fp32 and normalises the next
  // layer's input in the same launch (moe_forward_resnorm)
  float* cur = hA;
  void* xin = xn;
  void* xnext = w + r.xn2;
  for (int l = 0; l < n_target; ++l) {
    float* out = cur == hA ? hB : hA;
    if ((rc = moe_forward_resnorm(target_layers[l], xin, k + 1, cur, out, xnext, eps, stream))) return rc;
    cur = out;
    std::swap(xin, xnext);
  }
  e = lm_forward(lm, cur, true, k + 1, eps, target_logits, st);
  MCK(e, "mtp_round: LM head (verify rows)");
  // noisy rows for the heads, and the rows the drafts are read from
  float* rows = reinterpret_cast<float*>(w + r.rows);
  if (act == MOE_ACT_BF16)
    e = launch_pdl(draft_rows_kernel<2>, k * k, 256, 0, st, (const float*)cur, noise, k, H, eps, (void*)(w + r.hin),
                   rows);
  else
    e = launch_pdl(draft_rows_kernel<4>, k * k, 256, 0, st, (const float*)cur, noise, k, H, eps, (void*)(w + r.hin),
                   rows);
  MCK(e, "mtp_round: draft rows");
  uint8_t* hout = head_out ? static_cast<uint8_t*>(head_out) : w + r.hout;
  for (int j = 0; j < k; ++j) {
    const size_t o = (size_t)j * k * H * esz;
    if ((rc = moe_forward(draft_heads[j], w + r.hin + o, j + 1, hout + o, stream))) return rc;
  }
  float* dlog = draft_logits ? draft_logits : reinterpret_cast<float*>(w + r.dlog);
  e = lm_forward(lm, rows, true, k, eps, dlog, st);
  MCK(e, "mtp_round: LM head (draft rows)");
  float* dprob = reinterpret_cast<float*>(w + r.dprob);
  e = launch_pdl(argmax_rows_kernel, k, kArgThreads, 0, st, (const float*)dlog, V, draft_ids, dprob);
  MCK(e, "mtp_round: draft argmax");
  e = accept_launch_cut(draft_ids, k, target_logits, V, dprob, p_min, out_n_accepted, out_next_token, w + r.acc, st);
  MCK(e, "mtp_round: acceptance");
  return MOE_OK;
}

int mtp_round_hidden(const void* workspace, size_t workspace_bytes, int32_t H, int32_t k, int32_t V, int32_t act_dtype,
                     int32_t n_target, float* h_out, void* stream) {
  if (!workspace || !h_out) return set_error(MOE_EINVAL, "mtp_round_hidden: NULL argument");
  if (n_target < 0) return set_error(MOE_EINVAL, "mtp_round_hidden: n_target < 0");
  const size_t need = mtp_round_workspace_bytes(H, k, V, act_dtype);
  if (need == 0) return set_error(MOE_EINVAL, "mtp_round_hidden: H / k / V / act_dtype outside the round's ranges");
  if (workspace_bytes < need) return set_error(MOE_EINVAL, "mtp_round_hidden: workspace %zu bytes, need %zu", workspace_bytes, need);
  const RoundLayout r = round_layout(H, k, V, act_dtype);
  // h_0 is written to hA and each target layer moves it to the other buffer
  const uint8_t* src = static_cast<const uint8_t*>(workspace) + (n_target % 2 == 0 ? r.hA : r.hB);
  MCK(cudaMemcpyAsync(h_out, src, (size_t)(k + 1) * H * 4, cudaMemcpyDeviceToDevice, static_cast<cudaStream_t>(stream)),
      "mtp_round_hidden: copy");
  return MOE_OK;
}

}  // extern "C"
