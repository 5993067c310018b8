// small_t.cu -- the fused MoE layer for the MTP verify batch (1 <= T <= 8).
//
// One persistent kernel per forward, one CTA per SM.  Warp 8 (one thread) is
// a producer that claims tiles from a global queue and streams each tile's
// weight chunks, plus the activation records they need, into a ring of
// shared-memory stages with 1-D TMA bulk copies.  Warps 0-7 consume: lane =
// weight row, warp = a slice of the chunk's 32-column blocks.
//
// Tile order in the queue (each kind only waits on kinds before it, so every
// tile another tile waits for has already been claimed by a running CTA):
//   router tiles     32 experts x 256 columns; partial logits to global.  The
//                    tiles of row group 0 also convert x into activation
//                    records.  The last router tile to finish computes the
//                    routing (top-k, gates, permutation, expert work list).
//   shared gate/up   16 outputs x full K per tile, tokens of the shared expert
//   routed gate/up   same, per routed work entry (<= 4 tokens of one expert)
//   down tiles       32 outputs x full I per tile, per entry (shared first)
// Hand-offs use last-arriver counters: the last gate/up tile of an entry turns
// its SwiGLU outputs into activation records and publishes the entry; the last
// down tile of a 32-row block combines that block of y in slot order.  No
// floating-point atomics: every sum has a fixed order, so results are
// bit-reproducible.  Every spin-wait is bounded; on timeout the kernel sets
// the status word and drains its own copies before leaving.
//
// Arithmetic: weights enter as their integer codes; activations as block
// fixed point (32 values share a power-of-two scale, L bytes per value);
// dp4a gives exact integer block dot products, scaled once per block:
//   Q8_0 : sum_i d q_i v_i   = d * ascale * sum_i q_i X_i
//   Q4KS : sum_i (a q_i - b) v_i = a * ascale * sum_i q_i X_i - b * sumx
#include <cstdio>

#include "layer.cuh"

namespace moe {

enum TileKind : int { kRouter = 0, kGateUp = 1, kDown = 2, kEnd = 3 };

struct Desc {
  int kind, chunk, nch, M;
  int entry, rb, nbc, fmt;
  int slot0, n_ent, n_tiles_entry, rg;
  int ks, pad0, pad1, pad2;
};

struct SmemPlan {
  int ring, bars, descs, red, misc, flags, total;
};

__host__ __device__ inline SmemPlan smem_plan(int n_stages, int stage_bytes, int misc_bytes) {
  SmemPlan p;
  p.ring = 0;
  p.bars = n_stages * stage_bytes;
  p.descs = p.bars + 2 * n_stages * 8;
  p.red = p.descs + n_stages * (int)sizeof(Desc);
  p.red = (p.red + 15) & ~15;
  p.misc = p.red + kConsumerWarps * kMaxSmallT * 32 * 4;
  p.flags = p.misc + misc_bytes;
  p.total = p.flags + 64;
  return p;
}

// Records the first timeout: status[1] = wait site, status[2] = detail
// (tile, entry or stage), status[3] = CTA.
__device__ inline void record_timeout(int* status, int site, int detail) {
  if (atomicCAS(status, 0, kStatusTimeout) == 0) {
    status[1] = site;
    status[2] = detail;
    status[3] = blockIdx.x;
    __threadfence();
  }
}

enum WaitSite : int { kSiteRouting = 1, kSiteX = 2, kSiteEntry = 3, kSiteEmpty = 4, kSiteFull = 5, kSiteEnd = 6,
                      kSiteDrain = 7 };

// Bounded spin on a global flag (acquire).  Returns false on timeout.
__device__ inline bool wait_flag_geq(const int* p, int v, uint64_t limit_ns, int* status, int site, int detail) {
  if (ld_acquire(p) >= v) return true;
  const uint64_t t0 = globaltimer_ns();
  int ns = 32;
  while (true) {
    if (ld_acquire(p) >= v) return true;
    if (ld_acquire(status) != 0) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      record_timeout(status, site, detail);
      return false;
    }
    __nanosleep(ns);
    ns = min(ns * 2, 1024);
  }
}

__device__ inline bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, uint64_t limit_ns, int* status, int site,
                                         int detail) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(bar, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) {
      record_timeout(status, site, detail);
      return false;
    }
  }
  return true;
}

__device__ inline void entry_info(const SmallParams& P, int entry, Entry& en) {
  if (entry < P.n_sh) {
    en.e = -1;
    en.slot0 = P.T * P.k + kGroup * entry;
    en.M = min(kGroup, P.T - kGroup * entry);
    for (int m = 0; m < kGroup; ++m) en.tok[m] = kGroup * entry + m;
  } else {
    const int* src = reinterpret_cast<const int*>(P.entries + entry);
    en.e = __ldcg(src + 0);
    en.slot0 = __ldcg(src + 1);
    en.M = __ldcg(src + 2);
    for (int m = 0; m < kGroup; ++m) en.tok[m] = __ldcg(src + 3 + m);
  }
}

// ---------------------------------------------------------------------------
// producer
// ---------------------------------------------------------------------------
template <int L>
__device__ void producer_loop(const SmallParams& P, uint8_t* smem, const SmemPlan& plan) {
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + plan.bars);
  uint64_t* empty = full + P.n_stages;
  Desc* descs = reinterpret_cast<Desc*>(smem + plan.descs);
  constexpr int RB = rec_bytes(L);
  const int NR = P.n_rg * P.n_ks;
  const int NSG = P.n_sh * P.n_rb_sh;
  int s = 0;
  uint32_t ph = 0;
  int last_ph[8];
  for (int i = 0; i < 8; ++i) last_ph[i] = -1;
  bool ok = true;
  int n_rent = -1;

  while (ok) {
    const int t = atomicAdd(&P.sync->queue, 1);
    Desc d{};
    Entry en{};
    const uint8_t* wbase = nullptr;
    int64_t cbytes = 0;
    if (t < NR) {
      d.kind = kRouter;
      d.rg = t / P.n_ks;
      d.ks = t % P.n_ks;
      d.nch = 1;
      d.fmt = MOE_F32;
      d.nbc = kRouterKc / 32;
      wbase = P.router + (int64_t)t * chunk_bytes(MOE_F32, kRouterKc);
      cbytes = chunk_bytes(MOE_F32, kRouterKc);
    } else if (t < NR + NSG) {
      d.kind = kGateUp;
      d.entry = (t - NR) / P.n_rb_sh;
      d.rb = (t - NR) % P.n_rb_sh;
    } else {
      if (n_rent < 0) {
        if (!wait_flag_geq(&P.sync->routing_ready, 1, P.timeout_ns, P.status, kSiteRouting, t)) { ok = false; break; }
        fence_proxy_async_global();
        n_rent = __ldcg(&P.sync->n_rent);
      }
      const int A = NR + NSG;
      const int NG = n_rent * P.n_rb;
      const int ND = (P.n_sh + n_rent) * P.n_rbd;
      if (t < A + NG) {
        d.kind = kGateUp;
        d.entry = P.n_sh + (t - A) / P.n_rb;
        d.rb = (t - A) % P.n_rb;
      } else if (t < A + NG + ND) {
        d.kind = kDown;
        d.entry = (t - A - NG) / P.n_rbd;
        d.rb = (t - A - NG) % P.n_rbd;
      } else {
        break;  // queue exhausted
      }
    }
    if (d.kind != kRouter) {
      entry_info(P, d.entry, en);
      const bool sh = en.e < 0;
      d.M = en.M;
      d.slot0 = en.slot0;
      if (d.kind == kGateUp) {
        d.fmt = sh ? P.sfmt : P.fmt;
        d.nch = sh ? P.sgu_nch : P.gu_nch;
        const int kc = sh ? P.sgu_kc : P.gu_kc;
        d.nbc = kc / 32;
        cbytes = chunk_bytes(d.fmt, kc);
        wbase = (sh ? P.sgu : P.gu + (int64_t)en.e * P.gu_stride) + (int64_t)d.rb * d.nch * cbytes;
        d.n_tiles_entry = sh ? P.n_rb_sh : P.n_rb;
      } else {
        d.fmt = sh ? P.sfmt : P.fmt;
        d.nch = sh ? P.sdn_nch : P.dn_nch;
        const int kc = sh ? P.sdn_kc : P.dn_kc;
        d.nbc = kc / 32;
        cbytes = chunk_bytes(d.fmt, kc);
        wbase = (sh ? P.sdn : P.dn + (int64_t)en.e * P.dn_stride) + (int64_t)d.rb * d.nch * cbytes;
        d.n_ent = P.n_sh + n_rent;
      }
    }
    bool dep_ok = false;  // activation dependency satisfied for this tile
    for (int c = 0; c < d.nch && ok; ++c) {
      if (!mbar_wait_bounded(&empty[s], ph ^ 1u, P.timeout_ns, P.status, kSiteEmpty, t)) { ok = false; break; }
      d.chunk = c;
      uint8_t* stage = smem + plan.ring + s * P.stage_bytes;
      const uint32_t wb = (uint32_t)cbytes;
      const uint32_t ab = (d.kind == kRouter) ? 0u : (uint32_t)(d.M * d.nbc * RB);
      descs[s] = d;
      mbar_arrive_expect_tx(&full[s], wb + ab);
      bulk_g2s(stage, wbase + (int64_t)c * cbytes, wb, &full[s]);
      if (d.kind != kRouter) {
        if (!dep_ok) {
          if (d.kind == kGateUp) {
            // shared gate/up needs the x records; routed ones were gated by the routing flag
            if (en.e < 0) dep_ok = wait_flag_geq(&P.sync->x_done, P.n_ks, P.timeout_ns, P.status, kSiteX, t);
            else dep_ok = true;
          } else {
            dep_ok = wait_flag_geq(&P.entry_ready[d.entry], 1, P.timeout_ns, P.status, kSiteEntry,
                                   d.entry * 65536 + (t & 0xFFFF));
          }
        }
        if (dep_ok) fence_proxy_async_global();
        if (!dep_ok) {
          // keep the stage's byte count consistent: fill the activation part
          // with weight bytes again (the consumers see the status and stop)
          ok = false;
        }
        uint8_t* adst = stage + wb;
        const int kc = d.nbc * 32;
        for (int m = 0; m < d.M; ++m) {
          const uint8_t* src;
          if (!dep_ok) {
            src = wbase;  // harmless in-bounds bytes, only to complete the phase
          } else if (d.kind == kGateUp) {
            src = P.xrec + ((int64_t)en.tok[m] * (P.H / 32) + (int64_t)c * d.nbc) * RB;
          } else {
            src = P.hrec + ((int64_t)(en.slot0 + m) * (P.Imax / 32) + (int64_t)c * d.nbc) * RB;
          }
          (void)kc;
          bulk_g2s(adst + m * d.nbc * RB, src, (uint32_t)(d.nbc * RB), &full[s]);
        }
      }
      last_ph[s] = (int)ph;
      if (++s == P.n_stages) { s = 0; ph ^= 1u; }
    }
  }
  // end marker (or error): hand the consumers an END descriptor
  if (mbar_wait_bounded(&empty[s], ph ^ 1u, P.timeout_ns, P.status, kSiteEnd, s)) {
    Desc d{};
    d.kind = kEnd;
    descs[s] = d;
    mbar_arrive(&full[s]);
    // the consumers released this stage's previous fill, so its copies have
    // landed; the END arrival moved its barrier one phase on, so it must not
    // be waited for below
    last_ph[s] = -1;
  }
  // drain: every bulk copy this CTA issued must have landed before it exits
  // (a stage's barrier only advances past its last fill when that fill lands)
  for (int i = 0; i < P.n_stages; ++i)
    if (last_ph[i] >= 0) mbar_wait_bounded(&full[i], (uint32_t)last_ph[i], P.timeout_ns, P.status, kSiteDrain, i);
}

// ---------------------------------------------------------------------------
// consumer: chunk compute
// ---------------------------------------------------------------------------
template <int L>
__device__ __forceinline__ int block_dot_q8(uint4 q0, uint4 q1, const uint8_t* rec) {
  const uint4 a0 = *reinterpret_cast<const uint4*>(rec);
  const uint4 a1 = *reinterpret_cast<const uint4*>(rec + 16);
  int s0 = 0;
  s0 = dp4a_su(q0.x, a0.x, s0); s0 = dp4a_su(q0.y, a0.y, s0);
  s0 = dp4a_su(q0.z, a0.z, s0); s0 = dp4a_su(q0.w, a0.w, s0);
  s0 = dp4a_su(q1.x, a1.x, s0); s0 = dp4a_su(q1.y, a1.y, s0);
  s0 = dp4a_su(q1.z, a1.z, s0); s0 = dp4a_su(q1.w, a1.w, s0);
  return s0;
}
template <int L>
__device__ __forceinline__ int block_dot_q8_top(uint4 q0, uint4 q1, const uint8_t* rec) {
  const uint4 a0 = *reinterpret_cast<const uint4*>(rec);
  const uint4 a1 = *reinterpret_cast<const uint4*>(rec + 16);
  int s = 0;
  s = dp4a_ss(q0.x, a0.x, s); s = dp4a_ss(q0.y, a0.y, s);
  s = dp4a_ss(q0.z, a0.z, s); s = dp4a_ss(q0.w, a0.w, s);
  s = dp4a_ss(q1.x, a1.x, s); s = dp4a_ss(q1.y, a1.y, s);
  s = dp4a_ss(q1.z, a1.z, s); s = dp4a_ss(q1.w, a1.w, s);
  return s;
}

// sum over limbs of the block dot product, as float
template <int L>
__device__ __forceinline__ float limbs_q8(uint4 q0, uint4 q1, const uint8_t* rec) {
  if constexpr (L == 2) {
    const int s0 = block_dot_q8<L>(q0, q1, rec);
    const int s1 = block_dot_q8_top<L>(q0, q1, rec + 32);
    return (float)(s1 * 256 + s0);
  } else {
    const int s0 = block_dot_q8<L>(q0, q1, rec);
    const int s1 = block_dot_q8<L>(q0, q1, rec + 32);
    const int s2 = block_dot_q8<L>(q0, q1, rec + 64);
    const int s3 = block_dot_q8_top<L>(q0, q1, rec + 96);
    return fmaf((float)s3, 16777216.f, fmaf((float)s2, 65536.f, fmaf((float)s1, 256.f, (float)s0)));
  }
}

__device__ __forceinline__ int q4_dot(const uint32_t (&w)[8], const uint8_t* rec, bool top) {
  const uint4 a0 = *reinterpret_cast<const uint4*>(rec);
  const uint4 a1 = *reinterpret_cast<const uint4*>(rec + 16);
  int s = 0;
  if (!top) {
    s = dp4a_uu(w[0], a0.x, s); s = dp4a_uu(w[1], a0.y, s);
    s = dp4a_uu(w[2], a0.z, s); s = dp4a_uu(w[3], a0.w, s);
    s = dp4a_uu(w[4], a1.x, s); s = dp4a_uu(w[5], a1.y, s);
    s = dp4a_uu(w[6], a1.z, s); s = dp4a_uu(w[7], a1.w, s);
  } else {
    s = dp4a_us(w[0], a0.x, s); s = dp4a_us(w[1], a0.y, s);
    s = dp4a_us(w[2], a0.z, s); s = dp4a_us(w[3], a0.w, s);
    s = dp4a_us(w[4], a1.x, s); s = dp4a_us(w[5], a1.y, s);
    s = dp4a_us(w[6], a1.z, s); s = dp4a_us(w[7], a1.w, s);
  }
  return s;
}

template <int L>
__device__ __forceinline__ float limbs_q4(const uint32_t (&w)[8], const uint8_t* rec) {
  if constexpr (L == 2) {
    const int s0 = q4_dot(w, rec, false);
    const int s1 = q4_dot(w, rec + 32, true);
    return (float)(s1 * 256 + s0);
  } else {
    const int s0 = q4_dot(w, rec, false);
    const int s1 = q4_dot(w, rec + 32, false);
    const int s2 = q4_dot(w, rec + 64, false);
    const int s3 = q4_dot(w, rec + 96, true);
    return fmaf((float)s3, 16777216.f, fmaf((float)s2, 65536.f, fmaf((float)s1, 256.f, (float)s0)));
  }
}

__device__ __forceinline__ uint32_t field6(uint32_t w0, uint32_t w1, uint32_t w2, int f) {
  const int p = 6 * f;
  const int wi = p >> 5, sh = p & 31;
  const uint32_t lo = wi == 0 ? w0 : (wi == 1 ? w1 : w2);
  const uint32_t hi = wi == 0 ? w1 : (wi == 1 ? w2 : 0u);
  return __funnelshift_r(lo, hi, sh) & 63u;
}

template <int L>
__device__ __forceinline__ void gemv_chunk(const uint8_t* stage, const Desc& d, float (&acc)[kGroup]) {
  constexpr int RB = rec_bytes(L);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int nbc = d.nbc;
  const int nbw = (nbc + kConsumerWarps - 1) / kConsumerWarps;
  const int b0 = warp * nbw, b1 = min(nbc, b0 + nbw);
  const int M = d.M;
  const uint8_t* A = stage + chunk_bytes(d.fmt, nbc * 32);
  if (d.fmt == MOE_Q8_0) {
    const __half* sc = reinterpret_cast<const __half*>(stage + nbc * 1024);
    for (int b = b0; b < b1; ++b) {
      const uint4 q0 = *reinterpret_cast<const uint4*>(stage + ((b * 2 + 0) * 32 + lane) * 16);
      const uint4 q1 = *reinterpret_cast<const uint4*>(stage + ((b * 2 + 1) * 32 + lane) * 16);
      const float dq = __half2float(sc[b * 32 + lane]);
#pragma unroll
      for (int m = 0; m < kGroup; ++m) {
        if (m < M) {
          const uint8_t* rec = A + (m * nbc + b) * RB;
          const float asc = *reinterpret_cast<const float*>(rec + 32 * L);
          acc[m] = fmaf(dq * asc, limbs_q8<L>(q0, q1, rec), acc[m]);
        }
      }
    }
  } else {  // MOE_Q4KS
    const uint8_t* hdr_base = stage + nbc * 512;
    int cur_sb = -1;
    float dd = 0.f, dmin = 0.f;
    uint32_t f0 = 0, f1 = 0, f2 = 0;
    for (int b = b0; b < b1; ++b) {
      const int sb = b >> 3;
      if (sb != cur_sb) {
        const uint4 hd = *reinterpret_cast<const uint4*>(hdr_base + (sb * 32 + lane) * 16);
        dd = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu)));
        dmin = __half2float(__ushort_as_half((unsigned short)(hd.x >> 16)));
        f0 = hd.y; f1 = hd.z; f2 = hd.w;
        cur_sb = sb;
      }
      const int sidx = b & 7;
      const float a = dd * (float)field6(f0, f1, f2, sidx);
      const float bq = dmin * (float)field6(f0, f1, f2, 8 + sidx);
      const uint4 qv = *reinterpret_cast<const uint4*>(stage + (b * 32 + lane) * 16);
      uint32_t w[8];
      w[0] = qv.x & 0x0F0F0F0Fu; w[1] = (qv.x >> 4) & 0x0F0F0F0Fu;
      w[2] = qv.y & 0x0F0F0F0Fu; w[3] = (qv.y >> 4) & 0x0F0F0F0Fu;
      w[4] = qv.z & 0x0F0F0F0Fu; w[5] = (qv.z >> 4) & 0x0F0F0F0Fu;
      w[6] = qv.w & 0x0F0F0F0Fu; w[7] = (qv.w >> 4) & 0x0F0F0F0Fu;
#pragma unroll
      for (int m = 0; m < kGroup; ++m) {
        if (m < M) {
          const uint8_t* rec = A + (m * nbc + b) * RB;
          const float asc = *reinterpret_cast<const float*>(rec + 32 * L);
          const float sx = *reinterpret_cast<const float*>(rec + 32 * L + 4);
          acc[m] = fmaf(a * asc, limbs_q4<L>(w, rec), fmaf(-bq, sx, acc[m]));
        }
      }
    }
  }
}

// ---------------------------------------------------------------------------
// consumer: routing (last router tile)
// ---------------------------------------------------------------------------
__device__ void finalize_routing(const SmallParams& P, uint8_t* misc) {
  const int tid = threadIdx.x;
  const int T = P.T, E = P.E, k = P.k, Tk = P.T * P.k;
  float* lg = reinterpret_cast<float*>(misc);                       // [T*E]
  int* cnt = reinterpret_cast<int*>(misc + ((T * E * 4 + 15) & ~15)); // [E]
  int* sid = cnt + ((E + 3) & ~3);                                   // [Tk]
  float* sl = reinterpret_cast<float*>(sid + ((Tk + 3) & ~3));       // [Tk]
  int* sperm = reinterpret_cast<int*>(sl + ((Tk + 3) & ~3));         // [Tk]

  __threadfence();
  for (int i = tid; i < T * E; i += kConsumerWarps * 32) {
    const int t = i / E, e = i % E;
    float v = 0.f;
    for (int ks = 0; ks < P.n_ks; ++ks) v += __ldcg(&P.partials[((int64_t)ks * P.E_pad + e) * T + t]);
    if (P.router_b) v += P.router_b[e];
    lg[t * E + e] = v;
  }
  for (int e = tid; e < E; e += kConsumerWarps * 32) cnt[e] = 0;
  consumer_sync();

  // top-k per token (one warp per token): (value desc, index asc)
  const int lane = tid & 31, warp = tid >> 5;
  for (int t = warp; t < T; t += kConsumerWarps) {
    uint32_t chosen = 0;  // bit i <-> expert lane + 32 i
    for (int j = 0; j < k; ++j) {
      float best = -INFINITY;
      int bi = 0x7fffffff;
      for (int i = 0, e = lane; e < E; ++i, e += 32) {
        if (chosen & (1u << i)) continue;
        const float v = lg[t * E + e];
        if (v > best || (v == best && e < bi)) { best = v; bi = e; }
      }
#pragma unroll
      for (int o = 16; o; o >>= 1) {
        const float ob = __shfl_xor_sync(0xffffffffu, best, o);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, o);
        if (ob > best || (ob == best && oi < bi)) { best = ob; bi = oi; }
      }
      if ((bi & 31) == lane) chosen |= 1u << (bi >> 5);
      if (lane == 0) { sid[t * k + j] = bi; sl[t * k + j] = best; }
    }
    __syncwarp();
    if (lane < k) {
      const float l0 = sl[t * k];
      float sum = 0.f;
      for (int j = 0; j < k; ++j) sum += expf(sl[t * k + j] - l0);
      const float g = expf(sl[t * k + lane] - l0) / sum;
      P.gates[t * k + lane] = g;
      P.ids[t * k + lane] = sid[t * k + lane];
    }
  }
  consumer_sync();

  if (warp == 0) {
    // ranks of pairs within their expert (stable), histogram
    int rank[4], ep[4];
    for (int r = 0; r < 4; ++r) {
      const int p = lane + 32 * r;
      rank[r] = 0;
      ep[r] = -1;
      if (p < Tk) {
        ep[r] = sid[p];
        for (int q = 0; q < p; ++q) rank[r] += (sid[q] == ep[r]);
        atomicAdd(&cnt[ep[r]], 1);
      }
    }
    __syncwarp();
    // exclusive scans over experts: pair offsets, entry counts
    const int nper = (E + 31) / 32;
    const int e0 = lane * nper, e1 = min(E, e0 + nper);
    int sum_p = 0, sum_w = 0;
    for (int e = e0; e < e1; ++e) { sum_p += cnt[e]; sum_w += (cnt[e] + kGroup - 1) / kGroup; }
    int inc_p = sum_p, inc_w = sum_w;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int a = __shfl_up_sync(0xffffffffu, inc_p, o);
      const int b = __shfl_up_sync(0xffffffffu, inc_w, o);
      if (lane >= o) { inc_p += a; inc_w += b; }
    }
    int off = inc_p - sum_p, went = inc_w - sum_w;
    const int total_w = __shfl_sync(0xffffffffu, inc_w, 31);
    // offsets: reuse cnt[] as the running offset table
    for (int e = e0; e < e1; ++e) {
      const int c = cnt[e];
      P.offsets[e] = off;
      cnt[e] = off;  // now: start of expert e in perm
      if (c > 0) {
        for (int g = 0; g * kGroup < c; ++g) {
          int* dst = reinterpret_cast<int*>(P.entries + P.n_sh + went);
          dst[0] = e;
          dst[1] = off + g * kGroup;
          dst[2] = min(kGroup, c - g * kGroup);
          ++went;
        }
      }
      off += c;
    }
    if (lane == 31) P.offsets[E] = off;
    __syncwarp();
    for (int r = 0; r < 4; ++r) {
      const int p = lane + 32 * r;
      if (p < Tk) {
        const int slot = cnt[ep[r]] + rank[r];
        sperm[slot] = p;
        P.perm[slot] = p;
        P.pos[p] = slot;
      }
    }
    __syncwarp();
    // tokens of each routed entry
    for (int w = lane; w < total_w; w += 32) {
      int* dst = reinterpret_cast<int*>(P.entries + P.n_sh + w);
      const int slot0 = dst[1], M = dst[2];
      for (int m = 0; m < kGroup; ++m) dst[3 + m] = m < M ? sperm[slot0 + m] / k : 0;
    }
    if (lane == 0) P.sync->n_rent = total_w;
    __threadfence();
    __syncwarp();
    if (lane == 0) st_release(&P.sync->routing_ready, 1);
  }
}

// ---------------------------------------------------------------------------
// consumer loop
// ---------------------------------------------------------------------------
template <int L>
__device__ void consumer_loop(const SmallParams& P, uint8_t* smem, const SmemPlan& plan) {
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + plan.bars);
  uint64_t* empty = full + P.n_stages;
  const Desc* descs = reinterpret_cast<const Desc*>(smem + plan.descs);
  float* red = reinterpret_cast<float*>(smem + plan.red);  // [8 warps][8][32]
  uint8_t* misc = smem + plan.misc;
  int* flags = reinterpret_cast<int*>(smem + plan.flags);
  constexpr int RB = rec_bytes(L);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = P.T;
  int s = 0;
  uint32_t ph = 0;
  float acc[kGroup] = {0.f, 0.f, 0.f, 0.f};
  float racc[kMaxSmallT];

  while (true) {
    if (!mbar_wait_bounded(&full[s], ph, P.timeout_ns, P.status, kSiteFull, s)) break;
    const Desc d = descs[s];
    if (d.kind == kEnd) break;
    const uint8_t* stage = smem + plan.ring + s * P.stage_bytes;

    if (d.kind == kRouter) {
      // stage x[:, 256-column slice] as fp32
      float* xs = reinterpret_cast<float*>(misc);  // [T][256]
      const int col0 = d.ks * kRouterKc;
      for (int t = 0; t < T; ++t) {
        float v;
        if constexpr (L == 2) v = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(P.x)[(int64_t)t * P.H + col0 + tid]);
        else v = reinterpret_cast<const float*>(P.x)[(int64_t)t * P.H + col0 + tid];
        xs[t * kRouterKc + tid] = v;
      }
      consumer_sync();
      if (d.rg == 0) {
        // x slice -> activation records (warp w: block ks*8 + w)
        for (int t = 0; t < T; ++t)
          write_record<L>(xs[t * kRouterKc + warp * 32 + lane],
                          P.xrec + ((int64_t)t * (P.H / 32) + d.ks * 8 + warp) * RB);
        __threadfence();
        fence_proxy_async_global();
      }
      for (int t = 0; t < kMaxSmallT; ++t) racc[t] = 0.f;
      for (int k4 = warp * 8; k4 < warp * 8 + 8; ++k4) {
        const float4 w = *reinterpret_cast<const float4*>(stage + (k4 * 32 + lane) * 16);
#pragma unroll
        for (int t = 0; t < kMaxSmallT; ++t) {
          if (t < T) {
            const float4 xv = *reinterpret_cast<const float4*>(xs + t * kRouterKc + k4 * 4);
            racc[t] = fmaf(w.x, xv.x, fmaf(w.y, xv.y, fmaf(w.z, xv.z, fmaf(w.w, xv.w, racc[t]))));
          }
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
      for (int t = 0; t < kMaxSmallT; ++t)
        if (t < T) red[(warp * kMaxSmallT + t) * 32 + lane] = racc[t];
      consumer_sync();
      if (tid < T * 32) {
        const int t = tid >> 5, r = tid & 31;
        float v = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) v += red[(w * kMaxSmallT + t) * 32 + r];
        const int e = d.rg * 32 + r;
        P.partials[((int64_t)d.ks * P.E_pad + e) * T + t] = v;
      }
      __threadfence();
      consumer_sync();
      if (tid == 0) {
        if (d.rg == 0) atomicAdd(&P.sync->x_done, 1);
        const int old = atomicAdd(&P.sync->router_done, 1);
        flags[0] = (old == P.n_rg * P.n_ks - 1);
      }
      consumer_sync();
      if (flags[0]) finalize_routing(P, misc);
      consumer_sync();
    } else {
      if (d.chunk == 0)
        for (int m = 0; m < kGroup; ++m) acc[m] = 0.f;
      gemv_chunk<L>(stage, d, acc);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      if (d.chunk == d.nch - 1) {
        for (int m = 0; m < kGroup; ++m) red[(warp * kMaxSmallT + m) * 32 + lane] = acc[m];
        consumer_sync();
        if (d.kind == kGateUp) {
          const bool sh = d.entry < P.n_sh;
          if (tid < 16 * d.M) {
            const int i = tid & 15, m = tid >> 4;
            float g = 0.f, u = 0.f;
            for (int w = 0; w < kConsumerWarps; ++w) {
              g += red[(w * kMaxSmallT + m) * 32 + i];
              u += red[(w * kMaxSmallT + m) * 32 + 16 + i];
            }
            const float hv = g / (1.f + expf(-g)) * u;
            P.h[(int64_t)(d.slot0 + m) * P.Imax + d.rb * 16 + i] = hv;
          }
          __threadfence();
          consumer_sync();
          if (tid == 0) {
            const int old = atomicAdd(&P.gu_cnt[d.entry], 1);
            flags[0] = (old == d.n_tiles_entry - 1);
          }
          consumer_sync();
          if (flags[0]) {
            __threadfence();
            const int Ie = sh ? P.Ish : P.I;
            const int nblk = Ie / 32;
            for (int wi = warp; wi < d.M * nblk; wi += kConsumerWarps) {
              const int m = wi / nblk, b = wi % nblk;
              const float v = __ldcg(&P.h[(int64_t)(d.slot0 + m) * P.Imax + b * 32 + lane]);
              write_record<L>(v, P.hrec + ((int64_t)(d.slot0 + m) * (P.Imax / 32) + b) * RB);
            }
            __threadfence();
            fence_proxy_async_global();
            consumer_sync();
            if (tid == 0) st_release(&P.entry_ready[d.entry], 1);
          }
        } else {  // kDown
          if (tid < 32 * d.M) {
            const int r = tid & 31, m = tid >> 5;
            float v = 0.f;
            for (int w = 0; w < kConsumerWarps; ++w) v += red[(w * kMaxSmallT + m) * 32 + r];
            P.z[(int64_t)(d.slot0 + m) * P.H + d.rb * 32 + r] = v;
          }
          __threadfence();
          consumer_sync();
          if (tid == 0) {
            const int old = atomicAdd(&P.d_cnt[d.rb], 1);
            flags[0] = (old == d.n_ent - 1);
          }
          consumer_sync();
          if (flags[0]) {
            __threadfence();
            const int k = P.k;
            if (tid < T * 32) {
              const int t = tid >> 5, r = tid & 31;
              const int hh = d.rb * 32 + r;
              float v = 0.f;
              for (int j = 0; j < k; ++j) {
                const float g = __ldcg(&P.gates[t * k + j]);
                const int sl = __ldcg(&P.pos[t * k + j]);
                v = fmaf(g, __ldcg(&P.z[(int64_t)sl * P.H + hh]), v);
              }
              if (P.n_sh > 0) v += __ldcg(&P.z[(int64_t)(T * k + t) * P.H + hh]);
              if constexpr (L == 2) reinterpret_cast<__nv_bfloat16*>(P.y)[(int64_t)t * P.H + hh] = __float2bfloat16_rn(v);
              else reinterpret_cast<float*>(P.y)[(int64_t)t * P.H + hh] = v;
            }
          }
        }
        consumer_sync();
      }
    }
    if (++s == P.n_stages) { s = 0; ph ^= 1u; }
  }
}

template <int L>
__global__ void __launch_bounds__(kThreads, 1) moe_small_t_kernel(const __grid_constant__ SmallParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SmemPlan plan = smem_plan(P.n_stages, P.stage_bytes, P.misc_bytes);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + plan.bars);
  uint64_t* empty = full + P.n_stages;
  int* flags = reinterpret_cast<int*>(smem + plan.flags);
  if (threadIdx.x == 0) {
    for (int i = 0; i < P.n_stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5;
  if (warp == kConsumerWarps) {
    if ((threadIdx.x & 31) == 0) producer_loop<L>(P, smem, plan);
  } else {
    consumer_loop<L>(P, smem, plan);
  }

  // the last CTA out resets the cross-CTA counters for the next launch
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    const int old = atomicAdd(&P.sync->exit_cnt, 1);
    flags[1] = (old == (int)gridDim.x - 1);
  }
  __syncthreads();
  if (flags[1]) {
    __threadfence();
    for (int i = threadIdx.x; i < P.w_max; i += blockDim.x) {
      P.gu_cnt[i] = 0;
      P.entry_ready[i] = 0;
    }
    for (int i = threadIdx.x; i < P.n_rbd; i += blockDim.x) P.d_cnt[i] = 0;
    if (threadIdx.x == 0) {
      P.sync->queue = 0;
      P.sync->router_done = 0;
      P.sync->x_done = 0;
      P.sync->routing_ready = 0;
      P.sync->n_rent = 0;
      P.sync->exit_cnt = 0;
    }
    __threadfence();
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
int small_t_smem_bytes(const SmallParams& P) {
  return smem_plan(P.n_stages, P.stage_bytes, P.misc_bytes).total;
}

cudaError_t small_t_configure(int L, int smem_bytes) {
  if (L == 2)
    return cudaFuncSetAttribute(moe_small_t_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  return cudaFuncSetAttribute(moe_small_t_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

cudaError_t small_t_launch(const SmallParams& P, int L, int grid, int smem_bytes, cudaStream_t st) {
  if (L == 2) moe_small_t_kernel<2><<<grid, kThreads, smem_bytes, st>>>(P);
  else moe_small_t_kernel<4><<<grid, kThreads, smem_bytes, st>>>(P);
  return cudaGetLastError();
}

}  // namespace moe
