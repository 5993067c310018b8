// api.cu -- the extern "C" entry points of include/moe_layer.h.
#include <algorithm>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>

#include "layer.cuh"

namespace moe {
cudaError_t repack_matrix(int fmt, const uint8_t* src, uint8_t* dst, int rows, int K, int rows_per_tile, int lr_off,
                          Chunking ch, cudaStream_t st);
cudaError_t repack_router(const float* src, float* dst, int E, int E_pad, int H, cudaStream_t st);
cudaError_t quantize_launch(int fmt, const float* w, int64_t rows, int64_t cols, void* out, cudaStream_t st);
size_t accept_workspace_bytes(int k, int V);
cudaError_t accept_launch(const int32_t* draft, int k, const float* logits, int V, int32_t* out_n, int32_t* out_next,
                          void* ws, cudaStream_t st);
size_t accept_static_bytes();
cudaError_t accept_static_scratch(void** out);
int small_t_smem_bytes(const SmallParams& P);
int finalize_misc_bytes(int T, int E, int k);
cudaError_t small_t_configure(int L, int smem_bytes);
cudaError_t small_t_launch(const SmallParams& P, int L, int grid, int smem_bytes, cudaStream_t st);
cudaError_t small_t_init_logit_sums(const SmallParams& P, long long* lfx0, cudaStream_t st);
bool large_t_enabled(const moe_layer* L);
cudaError_t large_t_alloc(moe_layer* L);
cudaError_t large_t_repack(moe_layer* L, int which, int e, const uint8_t* src, cudaStream_t st);
cudaError_t large_t_repack_router(moe_layer* L, const float* src, cudaStream_t st);
size_t large_t_weight_bytes(const moe_layer* L);
size_t large_t_workspace_bytes(const moe_layer* L);
int* large_t_status_word(const moe_layer* L);
int* large_t_counters(const moe_layer* L);
cudaError_t large_t_forward(moe_layer* L, const void* x, int T, void* y, bool residual, cudaStream_t st);
cudaError_t large_t_get_routing(moe_layer* L, int32_t* ids, float* gates, int32_t* offsets, int32_t* perm,
                                cudaStream_t st);
void large_t_release(moe_layer* L);
}  // namespace moe

using namespace moe;

namespace {

thread_local std::string g_err = "no error";

int fail(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

}  // namespace

int moe::set_error(int code, const char* fmt, ...) {
  char buf[512];
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(buf, sizeof buf, fmt, ap);
  va_end(ap);
  g_err = buf;
  return code;
}

namespace {

int cuda_fail(cudaError_t e, const char* what) {
  return fail(e == cudaErrorMemoryAllocation ? MOE_ENOMEM : MOE_ECUDA, "%s: %s", what, cudaGetErrorString(e));
}

#define CK(call, what)                           \
  do {                                           \
    cudaError_t e_ = (call);                     \
    if (e_ != cudaSuccess) return cuda_fail(e_, what); \
  } while (0)

size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

bool is_device_ptr(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return false;
  }
  return a.type == cudaMemoryTypeDevice || a.type == cudaMemoryTypeManaged;
}

size_t fmt_bytes(int fmt, int64_t rows, int64_t cols) {
  if (rows <= 0 || cols <= 0) return 0;
  if (fmt == MOE_Q8_0) return cols % 32 ? 0 : (size_t)rows * (size_t)(cols / 32) * 34;
  if (fmt == MOE_Q4KS) return cols % 256 ? 0 : (size_t)rows * (size_t)(cols / 256) * 144;
  if (fmt == MOE_F32) return (size_t)rows * (size_t)cols * 4;
  return 0;
}

int check_tensor(const moe_tensor& t, int64_t rows, int64_t cols, bool quant, const char* name) {
  if (t.reserved != 0) return fail(MOE_EINVAL, "%s: reserved field must be 0", name);
  if (t.rows != rows || t.cols != cols)
    return fail(MOE_EINVAL, "%s: shape [%lld, %lld], expected [%lld, %lld]", name, (long long)t.rows,
                (long long)t.cols, (long long)rows, (long long)cols);
  if (quant && t.fmt != MOE_Q8_0 && t.fmt != MOE_Q4KS)
    return fail(MOE_EFORMAT, "%s: format %d not supported (Q8_0 or Q4KS)", name, t.fmt);
  if (!quant && t.fmt != MOE_F32) return fail(MOE_EFORMAT, "%s: must be MOE_F32", name);
  const size_t nb = fmt_bytes(t.fmt, rows, cols);
  if (nb == 0) return fail(MOE_EFORMAT, "%s: %lld columns do not fit format %d", name, (long long)cols, t.fmt);
  if (t.nbytes != nb) return fail(MOE_EINVAL, "%s: nbytes %zu, expected %zu", name, t.nbytes, nb);
  if (!t.data) return fail(MOE_EINVAL, "%s: data is NULL", name);
  return MOE_OK;
}

// Copies a source tensor to a device staging buffer when it lives on the host.
struct Stager {
  uint8_t* buf = nullptr;
  size_t cap = 0;
  ~Stager() {
    if (buf) cudaFree(buf);
  }
  int get(const void* src, size_t n, cudaStream_t st, const uint8_t** out) {
    if (is_device_ptr(src)) {
      *out = static_cast<const uint8_t*>(src);
      return MOE_OK;
    }
    if (n > cap) {
      CK(cudaStreamSynchronize(st), "staging sync");
      if (buf) cudaFree(buf);
      buf = nullptr;
      CK(cudaMalloc(&buf, n), "staging alloc");
      cap = n;
    }
    CK(cudaMemcpyAsync(buf, src, n, cudaMemcpyHostToDevice, st), "staging copy");
    *out = buf;
    return MOE_OK;
  }
};

void free_layer(moe_layer* L) {
  if (!L) return;
  large_t_release(L);
  cudaFree(L->router);
  cudaFree(L->router_b);
  cudaFree(L->gu);
  cudaFree(L->dn);
  cudaFree(L->sgu);
  cudaFree(L->sdn);
  cudaFree(L->ws);
  delete L;
}

int64_t tile_bytes_total(int fmt, int rows_tiles, Chunking ch) {
  return (int64_t)rows_tiles * ch.n * chunk_bytes(fmt, ch.Kc);
}

}  // namespace

extern "C" {

const char* moe_last_error(void) { return g_err.c_str(); }

size_t moe_quantized_bytes(int32_t fmt, int64_t rows, int64_t cols) {
  if (fmt != MOE_Q8_0 && fmt != MOE_Q4KS) return 0;
  return fmt_bytes(fmt, rows, cols);
}

int moe_quantize(int32_t fmt, const float* w, int64_t rows, int64_t cols, void* out, void* stream) {
  if (fmt != MOE_Q8_0 && fmt != MOE_Q4KS) return fail(MOE_EFORMAT, "moe_quantize: format %d", fmt);
  if (!w || !out) return fail(MOE_EINVAL, "moe_quantize: NULL pointer");
  if (fmt_bytes(fmt, rows, cols) == 0) return fail(MOE_EFORMAT, "moe_quantize: shape does not fit format");
  if ((reinterpret_cast<uintptr_t>(w) & 3) != 0) return fail(MOE_EINVAL, "moe_quantize: w not 4-byte aligned");
  CK(quantize_launch(fmt, w, rows, cols, out, static_cast<cudaStream_t>(stream)), "moe_quantize launch");
  return MOE_OK;
}

int moe_layer_create(const moe_layer_desc* d, void* stream, moe_layer** out) {
  if (!d || !out) return fail(MOE_EINVAL, "moe_layer_create: NULL argument");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (d->H <= 0 || d->H % 256 || d->H > 128 * kMaxDownTiles)
    return fail(MOE_EINVAL, "H=%d must be a positive multiple of 256, at most %d", d->H, 128 * kMaxDownTiles);
  if (d->E < 1 || d->E > 1024) return fail(MOE_EINVAL, "E=%d out of range 1..1024", d->E);
  if (d->top_k < 1 || d->top_k > std::min(d->E, 16)) return fail(MOE_EINVAL, "top_k=%d out of range", d->top_k);
  if (d->I <= 0 || d->I % 32) return fail(MOE_EINVAL, "I=%d must be a positive multiple of 32", d->I);
  if (d->I_shared < 0 || d->I_shared % 32) return fail(MOE_EINVAL, "I_shared=%d must be a multiple of 32", d->I_shared);
  if (d->T_max < 1 || d->T_max > 8192) return fail(MOE_EINVAL, "T_max=%d out of range 1..8192", d->T_max);
  if (d->act_dtype != MOE_ACT_BF16 && d->act_dtype != MOE_ACT_F32)
    return fail(MOE_EINVAL, "act_dtype=%d", d->act_dtype);
  if (!d->gate || !d->up || !d->down) return fail(MOE_EINVAL, "gate/up/down descriptor arrays are NULL");
  // the routed experts held (expert parallelism)
  const int e0 = d->expert_begin, n_e = d->expert_count == 0 ? d->E : d->expert_count;
  if (d->expert_count < 0 || e0 < 0 || (d->expert_count == 0 && e0 != 0) || n_e < 1 || e0 + n_e > d->E)
    return fail(MOE_EINVAL, "expert range [%d, %d + %d) outside 0..E=%d (expert_count 0 means all E from 0)", e0, e0,
                d->expert_count, d->E);
  if (d->T_max > kMaxSmallT) {
    // the tensor-core path: 128-row weight tiles, 64-column K-blocks, bf16 operands
    if (d->act_dtype != MOE_ACT_BF16)
      return fail(MOE_EINVAL, "T_max=%d: batches above %d tokens run in bf16 only (act_dtype must be MOE_ACT_BF16)",
                  d->T_max, kMaxSmallT);
    if (d->I % 64 || d->I_shared % 64)
      return fail(MOE_EINVAL, "T_max=%d: I=%d and I_shared=%d must be multiples of 64 for batches above %d tokens",
                  d->T_max, d->I, d->I_shared, kMaxSmallT);
  }
  int rc;
  if ((rc = check_tensor(d->router_w, d->E, d->H, false, "router_w"))) return rc;
  const bool has_bias = d->router_b.data != nullptr;
  if (has_bias && (rc = check_tensor(d->router_b, 1, d->E, false, "router_b"))) return rc;
  const int fmt = d->gate[0].fmt;
  for (int e = 0; e < n_e; ++e) {
    char nm[64];
    snprintf(nm, sizeof nm, "gate[%d]", e);
    if ((rc = check_tensor(d->gate[e], d->I, d->H, true, nm))) return rc;
    snprintf(nm, sizeof nm, "up[%d]", e);
    if ((rc = check_tensor(d->up[e], d->I, d->H, true, nm))) return rc;
    snprintf(nm, sizeof nm, "down[%d]", e);
    if ((rc = check_tensor(d->down[e], d->H, d->I, true, nm))) return rc;
    if (d->gate[e].fmt != fmt || d->up[e].fmt != fmt || d->down[e].fmt != fmt)
      return fail(MOE_EFORMAT, "expert %d: all routed matrices must share one format", e);
  }
  const bool has_sh = d->I_shared > 0;
  int sfmt = fmt;
  if (has_sh) {
    if ((rc = check_tensor(d->sh_gate, d->I_shared, d->H, true, "sh_gate"))) return rc;
    if ((rc = check_tensor(d->sh_up, d->I_shared, d->H, true, "sh_up"))) return rc;
    if ((rc = check_tensor(d->sh_down, d->H, d->I_shared, true, "sh_down"))) return rc;
    sfmt = d->sh_gate.fmt;
    if (d->sh_up.fmt != sfmt || d->sh_down.fmt != sfmt)
      return fail(MOE_EFORMAT, "shared expert: all matrices must share one format");
  }

  moe_layer* L = new moe_layer();
  L->H = d->H; L->E = d->E; L->k = d->top_k; L->I = d->I; L->Ish = d->I_shared;
  L->T_max = d->T_max; L->act = d->act_dtype; L->fmt = fmt; L->sfmt = sfmt;
  L->e0 = e0; L->n_e = n_e;
  L->timeout_ns = d->wait_limit_us ? (uint64_t)d->wait_limit_us * 1000ull : 2000000000ull;
  struct Guard {
    moe_layer* L;
    bool keep = false;
    ~Guard() {
      if (!keep) free_layer(L);
    }
  } guard{L};

  CK(cudaGetDevice(&L->dev), "cudaGetDevice");
  CK(cudaDeviceGetAttribute(&L->num_sms, cudaDevAttrMultiProcessorCount, L->dev), "SM count");
  // chunk sizes: the largest that let the shared-memory ring hold two
  // stages as they usually come, and any stage at all.  A stage is one
  // weight chunk plus the activation records of its tokens.  Routed entries
  // of the verify batch almost always hold one token (T tokens spread over
  // T*k of E experts), so routed stages are double-buffered at one token and
  // only have to fit the ring once at kGroup tokens; the shared expert
  // always carries a full token group.
  int max_optin = 0;
  CK(cudaDeviceGetAttribute(&max_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, L->dev), "smem attr");
  const int L_limbs = d->act_dtype == MOE_ACT_BF16 ? 2 : 4;
  const int RB = rec_bytes(L_limbs);
  auto stage_need = [&](int f, Chunking ch, int tokens) {
    return chunk_bytes(f, ch.Kc) + (int64_t)tokens * (ch.Kc / 32) * RB;
  };
  int64_t stage = 0, single = 0;  // the double-buffered stage, the largest stage
  for (int shift = 0; shift < 6; ++shift) {
    L->gu_ch = choose_chunking(fmt, d->H, shift);
    L->dn_ch = choose_chunking(fmt, d->I, shift);
    if (L->gu_ch.n == 0 || L->dn_ch.n == 0) return fail(MOE_EFORMAT, "no chunking for format %d", fmt);
    if (has_sh) {
      L->sgu_ch = choose_chunking(sfmt, d->H, shift);
      L->sdn_ch = choose_chunking(sfmt, d->I_shared, shift);
      if (L->sgu_ch.n == 0 || L->sdn_ch.n == 0) return fail(MOE_EFORMAT, "no chunking for shared format %d", sfmt);
    }
    // a router stage: room for one tile's weights (512 columns) and its x slice
    stage = kRouterTileChunks * chunk_bytes(MOE_F32, kRouterCc) +
            (int64_t)std::min(d->T_max, kMaxSmallT) * kRouterTileChunks * kRouterCc * (L_limbs == 2 ? 2 : 4);
    single = stage;
    stage = std::max(stage, stage_need(fmt, L->gu_ch, 1));
    stage = std::max(stage, stage_need(fmt, L->dn_ch, 1));
    single = std::max({single, stage_need(fmt, L->gu_ch, kGroup), stage_need(fmt, L->dn_ch, kGroup)});
    if (has_sh) {
      stage = std::max({stage, stage_need(sfmt, L->sgu_ch, kGroup), stage_need(sfmt, L->sdn_ch, kGroup)});
      single = std::max(single, stage);
    }
    stage = align_up(stage, 128);
    single = align_up(single, 128);
    if (2 * stage + 40 * 1024 <= max_optin && single + 40 * 1024 <= max_optin) break;
  }
  const int n_rg = (d->E + 31) / 32, n_ks = d->H / kRouterKc;
  const int E_pad = n_rg * 32;
  L->gu_stride = tile_bytes_total(fmt, d->I / 16, L->gu_ch);
  L->dn_stride = tile_bytes_total(fmt, d->H / 32, L->dn_ch);
  const size_t router_bytes = (size_t)E_pad * d->H * 4;
  CK(cudaMalloc(&L->router, router_bytes), "alloc router");
  if (has_bias) CK(cudaMalloc(&L->router_b, (size_t)d->E * 4), "alloc bias");
  CK(cudaMalloc(&L->gu, (size_t)L->gu_stride * n_e), "alloc gate/up");
  CK(cudaMalloc(&L->dn, (size_t)L->dn_stride * n_e), "alloc down");
  size_t sgu_b = 0, sdn_b = 0;
  if (has_sh) {
    sgu_b = tile_bytes_total(sfmt, d->I_shared / 16, L->sgu_ch);
    sdn_b = tile_bytes_total(sfmt, d->H / 32, L->sdn_ch);
    CK(cudaMalloc(&L->sgu, sgu_b), "alloc shared gate/up");
    CK(cudaMalloc(&L->sdn, sdn_b), "alloc shared down");
  }
  L->weight_bytes = router_bytes + (has_bias ? d->E * 4 : 0) + (size_t)(L->gu_stride + L->dn_stride) * n_e +
                    sgu_b + sdn_b;
  if (large_t_enabled(L)) {
    CK(large_t_alloc(L), "allocate the prefill-sized path");
    L->weight_bytes += large_t_weight_bytes(L);
  }
  const bool lt = L->lt != nullptr;

  // upload + repack
  Stager stg;
  const uint8_t* src = nullptr;
  if ((rc = stg.get(d->router_w.data, d->router_w.nbytes, st, &src))) return rc;
  CK(repack_router(reinterpret_cast<const float*>(src), reinterpret_cast<float*>(L->router), d->E, E_pad, d->H, st),
     "repack router");
  if (lt) CK(large_t_repack_router(L, reinterpret_cast<const float*>(src), st), "repack router (tensor-core path)");
  if (has_bias) {
    const cudaMemcpyKind kind = is_device_ptr(d->router_b.data) ? cudaMemcpyDeviceToDevice : cudaMemcpyHostToDevice;
    CK(cudaMemcpyAsync(L->router_b, d->router_b.data, (size_t)d->E * 4, kind, st), "copy bias");
  }
  for (int e = 0; e < n_e; ++e) {
    uint8_t* gu = L->gu + (int64_t)e * L->gu_stride;
    uint8_t* dn = L->dn + (int64_t)e * L->dn_stride;
    if ((rc = stg.get(d->gate[e].data, d->gate[e].nbytes, st, &src))) return rc;
    CK(repack_matrix(fmt, src, gu, d->I, d->H, 16, 0, L->gu_ch, st), "repack gate");
    if (lt) CK(large_t_repack(L, 0, e, src, st), "repack gate (tensor-core path)");
    if ((rc = stg.get(d->up[e].data, d->up[e].nbytes, st, &src))) return rc;
    CK(repack_matrix(fmt, src, gu, d->I, d->H, 16, 16, L->gu_ch, st), "repack up");
    if (lt) CK(large_t_repack(L, 1, e, src, st), "repack up (tensor-core path)");
    if ((rc = stg.get(d->down[e].data, d->down[e].nbytes, st, &src))) return rc;
    CK(repack_matrix(fmt, src, dn, d->H, d->I, 32, 0, L->dn_ch, st), "repack down");
    if (lt) CK(large_t_repack(L, 2, e, src, st), "repack down (tensor-core path)");
  }
  if (has_sh) {
    if ((rc = stg.get(d->sh_gate.data, d->sh_gate.nbytes, st, &src))) return rc;
    CK(repack_matrix(sfmt, src, L->sgu, d->I_shared, d->H, 16, 0, L->sgu_ch, st), "repack shared gate");
    if (lt) CK(large_t_repack(L, 3, 0, src, st), "repack shared gate (tensor-core path)");
    if ((rc = stg.get(d->sh_up.data, d->sh_up.nbytes, st, &src))) return rc;
    CK(repack_matrix(sfmt, src, L->sgu, d->I_shared, d->H, 16, 16, L->sgu_ch, st), "repack shared up");
    if (lt) CK(large_t_repack(L, 4, 0, src, st), "repack shared up (tensor-core path)");
    if ((rc = stg.get(d->sh_down.data, d->sh_down.nbytes, st, &src))) return rc;
    CK(repack_matrix(sfmt, src, L->sdn, d->H, d->I_shared, 32, 0, L->sdn_ch, st), "repack shared down");
    if (lt) CK(large_t_repack(L, 5, 0, src, st), "repack shared down (tensor-core path)");
  }

  // small-T workspace
  const int Tm = std::min(d->T_max, kMaxSmallT);
  const int k = d->top_k;
  const int P = Tm * k + Tm;
  const int Imax = std::max(d->I, d->I_shared);
  const int w_max = (Tm + kGroup - 1) / kGroup + Tm * k;
  const int n_dt = d->H / 128;
  SmallParams& sp = L->sp;
  sp = SmallParams{};
  sp.H = d->H; sp.E = d->E; sp.k = k; sp.I = d->I; sp.Ish = d->I_shared;
  sp.e0 = e0; sp.n_e = n_e;
  sp.act_f32 = d->act_dtype == MOE_ACT_F32 ? 1 : 0;
  sp.n_rg = n_rg; sp.n_ks = n_ks; sp.n_rc = d->H / kRouterCc;
  sp.n_kt = (sp.n_rc + kRouterTileChunks - 1) / kRouterTileChunks; sp.n_gu = d->I / 32; sp.n_gu_sh = d->I_shared / 32; sp.n_dt = n_dt;
  sp.Imax = Imax; sp.E_pad = E_pad; sp.w_max = w_max;
  sp.router = L->router; sp.router_b = L->router_b;
  sp.gu = L->gu; sp.dn = L->dn; sp.sgu = L->sgu; sp.sdn = L->sdn;
  sp.gu_stride = L->gu_stride; sp.dn_stride = L->dn_stride;
  sp.fmt = fmt; sp.sfmt = sfmt;
  sp.gu_nch = L->gu_ch.n; sp.gu_kc = L->gu_ch.Kc; sp.dn_nch = L->dn_ch.n; sp.dn_kc = L->dn_ch.Kc;
  sp.sgu_nch = L->sgu_ch.n; sp.sgu_kc = L->sgu_ch.Kc; sp.sdn_nch = L->sdn_ch.n; sp.sdn_kc = L->sdn_ch.Kc;
  sp.timeout_ns = L->timeout_ns;

  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t o = off;
    off = align_up(off + bytes, 256);
    return o;
  };
  const size_t o_sync = take(sizeof(Sync));
  const size_t o_gucnt = take((size_t)w_max * 4);
  const size_t o_ready = take((size_t)w_max * 4);
  const size_t o_dcnt = take((size_t)n_dt * 4);
  const size_t o_lfx = take((size_t)E_pad * 8 * 8);  // the bias between launches (reset by the last block)
  const size_t counters_end = off;
  const size_t o_status = take(16);
  const size_t o_stamps = take(2 * kNumStamps * 8);
  const size_t o_lfx0 = take((size_t)E_pad * 8);
  const size_t o_ids = take((size_t)Tm * k * 4);
  const size_t o_gates = take((size_t)Tm * k * 4);
  const size_t o_pos = take((size_t)Tm * k * 4);
  const size_t o_offs = take((size_t)(d->E + 1) * 4);
  const size_t o_perm = take((size_t)Tm * k * 4);
  const size_t o_ent = take((size_t)w_max * sizeof(Entry));
  const size_t o_xrec = take((size_t)Tm * (d->H / 32) * RB);
  const size_t o_hrec = take((size_t)P * (Imax / 32) * RB);
  const size_t o_z = take((size_t)P * d->H * 4);
  const size_t o_ssq = take((size_t)kMaxSmallT * n_dt * 4);
  L->ws_bytes = off;
  CK(cudaMalloc(&L->ws, L->ws_bytes), "alloc workspace");
  CK(cudaMemsetAsync(L->ws, 0, L->ws_bytes, st), "zero workspace");
  uint8_t* w = static_cast<uint8_t*>(L->ws);
  sp.sync = reinterpret_cast<Sync*>(w + o_sync);
  sp.gu_cnt = reinterpret_cast<int*>(w + o_gucnt);
  sp.entry_ready = reinterpret_cast<int*>(w + o_ready);
  sp.d_cnt = reinterpret_cast<int*>(w + o_dcnt);
  sp.status = reinterpret_cast<int*>(w + o_status);
  sp.ssq = reinterpret_cast<float*>(w + o_ssq);
  sp.stamps = reinterpret_cast<unsigned long long*>(w + o_stamps);
  sp.lfx0 = reinterpret_cast<const long long*>(w + o_lfx0);
  sp.lfx = reinterpret_cast<long long*>(w + o_lfx);
  sp.ids = reinterpret_cast<int*>(w + o_ids);
  sp.gates = reinterpret_cast<float*>(w + o_gates);
  sp.pos = reinterpret_cast<int*>(w + o_pos);
  sp.offsets = reinterpret_cast<int*>(w + o_offs);
  sp.perm = reinterpret_cast<int*>(w + o_perm);
  sp.entries = reinterpret_cast<Entry*>(w + o_ent);
  sp.xrec = w + o_xrec;
  sp.hrec = w + o_hrec;
  sp.z = reinterpret_cast<float*>(w + o_z);
  (void)counters_end;

  sp.misc_bytes = (int)align_up((size_t)finalize_misc_bytes(Tm, d->E, k), 16);
  // every byte not needed elsewhere goes to the stage ring; it must hold at
  // least two of the largest stages
  sp.n_stages = kMaxSlots;
  sp.ring_bytes = 0;
  const int fixed = small_t_smem_bytes(sp);
  sp.ring_bytes = (int)((max_optin - fixed) / 128 * 128);
  if (sp.ring_bytes < 2 * stage || sp.ring_bytes < single)
    return fail(MOE_EINVAL, "layer shapes need more shared memory than the device has (stage %lld B, largest %lld B)",
                (long long)stage, (long long)single);
  L->smem_bytes = small_t_smem_bytes(sp);
  // the attribute belongs to the kernel, not to this layer: set it to the
  // device limit, which bounds every layer's plan
  CK(small_t_configure(L_limbs, max_optin), "configure small-T kernel");

  CK(small_t_init_logit_sums(sp, reinterpret_cast<long long*>(w + o_lfx0), st), "logit sums init");
  CK(cudaStreamSynchronize(st), "create sync");
  guard.keep = true;
  *out = L;
  g_err = "no error";
  return MOE_OK;
}

}  // extern "C"

namespace {
struct ResNorm {  // moe_forward_resnorm's outputs
  const float* h_in;
  float* h_out;
  void* xn;
  float eps;
};

int forward_impl(moe_layer* L, const void* x, int32_t T, void* y, void* stream, bool residual, bool out_f32,
                 const ResNorm* rn = nullptr) {
  if (!L) return fail(MOE_EINVAL, "moe_forward: NULL layer");
  if (T < 0 || T > L->T_max) return fail(MOE_EINVAL, "moe_forward: T=%d outside 0..%d", T, L->T_max);
  if (T == 0) return MOE_OK;
  if (!x || !y) return fail(MOE_EINVAL, "moe_forward: NULL x or y");
  if ((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(y)) & 15)
    return fail(MOE_EINVAL, "moe_forward: x and y must be 16-byte aligned");
  if (out_f32 && T > kMaxSmallT) return fail(MOE_EINVAL, "moe_forward_f32: T=%d above %d", T, kMaxSmallT);
  const size_t esz = L->act == MOE_ACT_BF16 ? 2 : 4;
  const uintptr_t xb = reinterpret_cast<uintptr_t>(x), yb = reinterpret_cast<uintptr_t>(y);
  const size_t nbx = (size_t)T * L->H * esz, nby = (size_t)T * L->H * (out_f32 ? 4 : esz);
  if (xb < yb + nby && yb < xb + nbx) return fail(MOE_EINVAL, "moe_forward: x and y overlap");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  L->last_T = T;
  if (T > kMaxSmallT) {
    CK(large_t_forward(L, x, T, y, residual, st), "moe_forward (tensor-core path)");
    return MOE_OK;
  }
  SmallParams P = L->sp;
  P.T = T;
  P.Tp = (T + 3) & ~3;
  P.n_sh = L->Ish > 0 ? (T + kGroup - 1) / kGroup : 0;
  P.x = x;
  P.y = y;
  P.residual = residual ? 1 : 0;
  P.out_f32 = out_f32 ? 1 : 0;
  P.h_in = nullptr;
  if (rn) {
    P.h_in = rn->h_in;
    P.h_out = rn->h_out;
    P.xn = rn->xn;
    P.eps = rn->eps;
  }
  P.ready_target = 1;
  if (L->inject == 1) {
    P.ready_target = 1 << 30;  // published as 1 + the routed entries: the routed tiles' wait runs out
    L->inject = 0;
  }
  CK(small_t_launch(P, L->act == MOE_ACT_BF16 ? 2 : 4, L->num_sms, L->smem_bytes, st), "moe_forward launch");
  return MOE_OK;
}
}  // namespace

extern "C" {

int moe_forward(moe_layer* L, const void* x, int32_t T, void* y, void* stream) {
  return forward_impl(L, x, T, y, stream, false, false);
}

int moe_forward_residual(moe_layer* L, const void* x, int32_t T, void* y, void* stream) {
  return forward_impl(L, x, T, y, stream, true, false);
}

int moe_forward_f32(moe_layer* L, const void* x, int32_t T, float* y, void* stream) {
  return forward_impl(L, x, T, y, stream, false, true);
}

int moe_forward_resnorm(moe_layer* L, const void* x, int32_t T, const float* h_in, float* h_out, void* xn, float eps,
                        void* stream) {
  if (!L) return fail(MOE_EINVAL, "moe_forward_resnorm: NULL layer");
  if (T < 0 || T > kMaxSmallT || T > L->T_max)
    return fail(MOE_EINVAL, "moe_forward_resnorm: T=%d outside 0..%d", T, std::min(kMaxSmallT, L->T_max));
  if (T == 0) return MOE_OK;
  if (!x || !h_in || !h_out || !xn) return fail(MOE_EINVAL, "moe_forward_resnorm: NULL argument");
  if (!(eps >= 0.f) || eps > 1e30f) return fail(MOE_EINVAL, "moe_forward_resnorm: eps must be finite and >= 0");
  if ((reinterpret_cast<uintptr_t>(h_in) | reinterpret_cast<uintptr_t>(h_out) | reinterpret_cast<uintptr_t>(xn)) & 15)
    return fail(MOE_EINVAL, "moe_forward_resnorm: h_in, h_out and xn must be 16-byte aligned");
  const size_t esz = L->act == MOE_ACT_BF16 ? 2 : 4, nh = (size_t)T * L->H * 4, nx = (size_t)T * L->H * esz;
  auto overlap = [](const void* a, size_t na, const void* b, size_t nb) {
    const uintptr_t pa = reinterpret_cast<uintptr_t>(a), pb = reinterpret_cast<uintptr_t>(b);
    return pa < pb + nb && pb < pa + na;
  };
  if (h_in != h_out && overlap(h_in, nh, h_out, nh))
    return fail(MOE_EINVAL, "moe_forward_resnorm: h_in and h_out overlap without being the same rows");
  if (overlap(x, nx, h_out, nh) || overlap(x, nx, xn, nx) || overlap(xn, nx, h_out, nh) || overlap(xn, nx, h_in, nh))
    return fail(MOE_EINVAL, "moe_forward_resnorm: x, xn and h_out must not overlap (nor xn and h_in)");
  const ResNorm rn{h_in, h_out, xn, eps};
  // y is not written in this mode; h_out stands in for it in the checks
  return forward_impl(L, x, T, h_out, stream, false, true, &rn);
}

int moe_get_routing(moe_layer* L, int32_t* ids, float* gates, int32_t* offsets, int32_t* perm, void* stream) {
  if (!L) return fail(MOE_EINVAL, "moe_get_routing: NULL layer");
  if (L->last_T <= 0) return fail(MOE_EINVAL, "moe_get_routing: no forward yet");
  if (L->last_T > kMaxSmallT) {
    CK(large_t_get_routing(L, ids, gates, offsets, perm, static_cast<cudaStream_t>(stream)), "moe_get_routing");
    return MOE_OK;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  const size_t Tk = (size_t)L->last_T * L->k;
  if (ids) CK(cudaMemcpyAsync(ids, L->sp.ids, Tk * 4, cudaMemcpyDeviceToDevice, st), "routing ids");
  if (gates) CK(cudaMemcpyAsync(gates, L->sp.gates, Tk * 4, cudaMemcpyDeviceToDevice, st), "routing gates");
  if (offsets)
    CK(cudaMemcpyAsync(offsets, L->sp.offsets, (size_t)(L->E + 1) * 4, cudaMemcpyDeviceToDevice, st), "offsets");
  if (perm) CK(cudaMemcpyAsync(perm, L->sp.perm, Tk * 4, cudaMemcpyDeviceToDevice, st), "routing perm");
  return MOE_OK;
}

int moe_layer_status(moe_layer* L, void* stream) {
  if (!L) return fail(MOE_EINVAL, "moe_layer_status: NULL layer");
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  CK(cudaStreamSynchronize(st), "status sync");
  int word[4] = {0, 0, 0, 0};
  CK(cudaMemcpy(word, L->sp.status, 16, cudaMemcpyDeviceToHost), "status read");
  if (word[0] != 0) {
    // clear the word and every cross-CTA counter so the next call starts clean
    const size_t counters = reinterpret_cast<uint8_t*>(L->sp.status) - static_cast<uint8_t*>(L->ws);
    CK(cudaMemset(L->ws, 0, counters + 16), "status reset");
    CK(small_t_init_logit_sums(L->sp, const_cast<long long*>(L->sp.lfx0), nullptr), "logit sums reset");
    CK(cudaDeviceSynchronize(), "status reset sync");
    static const char* sites[] = {"?",          "routing flag",        "x records",           "entry ready",
                                   "free stage", "full stage",          "end marker",          "copy drain",
                                   "free reduction slot", "full reduction slot", "router logit words"};
    const int site = (word[1] >= 0 && word[1] <= 10) ? word[1] : 0;
    return fail(MOE_ETIMEOUT, "a device-side wait timed out: %s (detail %d, block %d)", sites[site], word[2],
                word[3]);
  }
  if (int* lw = large_t_status_word(L)) {
    CK(cudaMemcpy(word, lw, 16, cudaMemcpyDeviceToHost), "status read");
    if (word[0] != 0) {
      CK(cudaMemset(lw, 0, 16), "status reset");
      CK(cudaMemset(large_t_counters(L), 0, 16 * 4), "counter reset");
      static const char* sites[] = {"?", "free stage", "full stage", "dequantised stage", "accumulator",
                                     "work item", "copy drain"};
      const int site = (word[1] >= 0 && word[1] <= 6) ? word[1] : 0;
      return fail(MOE_ETIMEOUT, "a device-side wait of the tensor-core path timed out: %s (detail %d, block %d)",
                  sites[site], word[2], word[3]);
    }
  }
  return MOE_OK;
}

int moe_layer_timeline(moe_layer* L, int64_t* out_ns, int32_t n, void* stream) {
  if (!L || !out_ns || n < 1) return fail(MOE_EINVAL, "moe_layer_timeline: NULL argument or n < 1");
  CK(cudaStreamSynchronize(static_cast<cudaStream_t>(stream)), "timeline sync");
  unsigned long long w[kNumStamps];
  CK(cudaMemcpy(w, L->sp.stamps + kNumStamps, sizeof w, cudaMemcpyDeviceToHost), "timeline read");
  auto at = [&](int i) -> int64_t {
    if (w[i] == 0ull) return -1;
    return (int64_t)(((kStampFirstMask >> i) & 1u) ? ~w[i] : w[i]);
  };
  const int64_t t0 = at(kTsStart);
  for (int i = 0; i < n; ++i) {
    const int64_t v = i < kNumStamps ? at(i) : -1;
    out_ns[i] = (v < 0 || t0 < 0) ? -1 : v - t0;
  }
  return MOE_OK;
}

int moe_layer_inject_timeout(moe_layer* L, int32_t site) {
  if (!L) return fail(MOE_EINVAL, "moe_layer_inject_timeout: NULL layer");
  if (site != 1) return fail(MOE_EINVAL, "moe_layer_inject_timeout: site %d (only 1 is defined)", site);
  L->inject = site;
  return MOE_OK;
}

size_t moe_layer_weight_bytes(const moe_layer* L) { return L ? L->weight_bytes : 0; }
size_t moe_layer_workspace_bytes(const moe_layer* L) { return L ? L->ws_bytes + large_t_workspace_bytes(L) : 0; }

void moe_layer_destroy(moe_layer* L) { free_layer(L); }

size_t mtp_verify_accept_workspace_bytes(int32_t k, int32_t V) {
  if (k < 0 || k > 15 || V < 1 || V > (1 << 24)) return 0;
  return accept_workspace_bytes(k, V);
}

int mtp_verify_accept(const int32_t* draft_ids, int32_t k, const float* logits, int32_t V, int32_t* out_n_accepted,
                      int32_t* out_next_token, void* workspace, size_t workspace_bytes, void* stream) {
  if (k < 0 || k > 15) return fail(MOE_EINVAL, "mtp_verify_accept: k=%d outside 0..15", k);
  if (V < 1 || V > (1 << 24)) return fail(MOE_EINVAL, "mtp_verify_accept: V=%d outside 1..2^24", V);
  if ((k > 0 && !draft_ids) || !logits || !out_n_accepted || !out_next_token || !workspace)
    return fail(MOE_EINVAL, "mtp_verify_accept: NULL pointer");
  if (reinterpret_cast<uintptr_t>(workspace) & 15)
    return fail(MOE_EINVAL, "mtp_verify_accept: workspace must be 16-byte aligned");
  if (workspace_bytes < accept_workspace_bytes(k, V))
    return fail(MOE_EINVAL, "mtp_verify_accept: workspace %zu bytes, need %zu", workspace_bytes,
                accept_workspace_bytes(k, V));
  CK(accept_launch(draft_ids, k, logits, V, out_n_accepted, out_next_token, workspace,
                   static_cast<cudaStream_t>(stream)),
     "mtp_verify_accept launch");
  return MOE_OK;
}

int mtp_verify_accept_noalloc(const int32_t* draft_ids, int32_t k, const float* logits, int32_t V,
                              int32_t* out_n_accepted, int32_t* out_next_token, void* stream) {
  if (k < 0 || k > 15) return fail(MOE_EINVAL, "mtp_verify_accept_noalloc: k=%d outside 0..15", k);
  if (V < 1 || V > (1 << 24)) return fail(MOE_EINVAL, "mtp_verify_accept_noalloc: V=%d outside 1..2^24", V);
  if ((k > 0 && !draft_ids) || !logits || !out_n_accepted || !out_next_token)
    return fail(MOE_EINVAL, "mtp_verify_accept_noalloc: NULL pointer");
  const size_t need = accept_workspace_bytes(k, V);
  if (need > accept_static_bytes())
    return fail(MOE_EINVAL,
                "mtp_verify_accept_noalloc: k=%d, V=%d needs %zu bytes of scratch but the static scratch holds "
                "%zu; use mtp_verify_accept with a caller workspace",
                k, V, need, accept_static_bytes());
  void* scratch = nullptr;
  CK(accept_static_scratch(&scratch), "mtp_verify_accept_noalloc: static scratch lookup");
  CK(accept_launch(draft_ids, k, logits, V, out_n_accepted, out_next_token, scratch,
                   static_cast<cudaStream_t>(stream)),
     "mtp_verify_accept_noalloc launch");
  return MOE_OK;
}

}  // extern "C"
