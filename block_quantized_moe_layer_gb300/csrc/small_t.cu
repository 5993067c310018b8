// small_t.cu -- the fused MoE layer for the MTP verify batch (1 <= T <= 8).
//
// One persistent kernel per forward, one CTA per SM, three warp roles:
//   producer (warp 8, one thread): claims tiles from a global queue (one claim
//     ahead) and streams each tile's weight chunks, plus the activation
//     records they need, into a ring of shared-memory stages with 1-D bulk
//     copies;
//   consumers (warps 0-7): lane = weight row, warp = a slice of the chunk's
//     32-column blocks; integer dot products per block;
//   epilogue (warp 9): takes each finished 32-row group's partial sums from a
//     small ring, reduces them and does the bookkeeping (SwiGLU and
//     activation records, down outputs, counters, the combine), so the
//     consumers never wait on global-memory round trips.
//
// Tile order in the queue (each kind only waits on kinds before it, so every
// tile another tile waits for has already been claimed by a running CTA):
//   x records        one per 512-column slice of x: all T tokens' activation
//                    records (one 32-column block per thread)
//   router tiles     32 experts x 512 columns; each adds its share of the
//                    logits to a global sum kept as exact 2^-32 fixed point
//                    (integer atomics, so the sum does not depend on the
//                    order of arrival).  The last router tile to finish
//                    computes the routing (top-k, gates, permutation, expert
//                    work entries).
//   shared gate/up   32 outputs (16+16 gate/up rows, twice) x full K
//   shared down      128 outputs x full I
//   routed gate/up   per routed work entry (<= 4 tokens of one expert)
//   routed down
// Hand-offs use last-arriver counters: the last gate/up tile of an entry
// publishes it (its activation records are complete); the last down tile of
// a 128-row block combines that block of y in slot order.  No floating-point
// atomics: every floating-point sum has a fixed order (the logits' integer
// sum has none to keep), so results are bit-reproducible.
// Every spin-wait is bounded; on timeout the kernel records where in the
// status word, drains its own copies and leaves.
//
// Arithmetic: weights enter as their integer codes; activations as block
// fixed point (32 values share a power-of-two scale, L bytes per value);
// dp4a gives exact integer block dot products, scaled once per block:
//   Q8_0 : sum_i d q_i v_i       = d * ascale * sum_i q_i X_i
//   Q4KS : sum_i (a q_i - b) v_i = a * ascale * sum_i q_i X_i - b * sumx
#include "layer.cuh"

namespace moe {

enum TileKind : int { kRouter = 0, kGateUp = 1, kDown = 2, kEnd = 3, kXRec = 4 };

struct Desc {
  int kind, chunk, nch, M;         // read by every consumer thread
  int nbc, fmt, rgks, off;         //   " (off = ring offset; rgks: router and x-record items: row
                                   //   group << 16 | chunk; gate/up and down: groups in the stage)
  int entry, rbt, group, ngroups;  // read by the epilogue warp
  int slot0, n_ent, n_tiles_entry, pad;
};

struct SmemPlan {
  int ring, bars, rbars, ebar, descs, metas, rred, red, misc, ecache, escr, pend, flags, total;
};

constexpr int kRedSlots = 4;
constexpr int kRedSlotBytes = kConsumerWarps * kRows * kGroup * 4;  // one 32-row group: [warp][row][token]

// The ring holds variable-size stages back to back (ring_bytes); n_slots
// descriptor slots, each with a full / empty barrier pair.
__host__ __device__ inline SmemPlan smem_plan(int n_stages, int ring_bytes, int misc_bytes, int w_max) {
  SmemPlan p;
  p.ring = 0;
  p.bars = ring_bytes;
  p.rbars = p.bars + 2 * n_stages * 8;
  p.ebar = p.rbars + 2 * kRedSlots * 8;  // the producer's work-entry copy
  p.descs = p.ebar + 16;
  p.metas = p.descs + n_stages * (int)sizeof(Desc);
  // the router's scratch (rred, misc) shares bytes with the epilogue ring: a
  // CTA's router tiles and the routing come before any of its gate/up or down
  // tiles, so the two are never live at once
  p.red = (p.metas + kRedSlots * (int)sizeof(Desc) + 15) & ~15;
  p.rred = p.red;
  p.misc = p.rred + kConsumerWarps * kMaxSmallT * 32 * 4;
  const int region = max(kRedSlots * kRedSlotBytes, kConsumerWarps * kMaxSmallT * 32 * 4 + misc_bytes);
  p.ecache = p.red + ((region + 15) & ~15);
  p.escr = p.ecache + ((w_max * (int)sizeof(Entry) + 15) & ~15);
  p.pend = p.escr + 2 * kMaxSmallT * kMaxTopK * 4;
  p.flags = p.pend + 4 * (1 + kMaxDownTiles);
  p.total = p.flags + 64;  // flags[0..3] and the producer's published-entry bits [4..11]
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
                      kSiteDrain = 7, kSiteRedEmpty = 8, kSiteRedFull = 9 };

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
    ns = min(ns * 2, 128);
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

__device__ inline void shared_entry(const SmallParams& P, int entry, Entry& en) {
  en.e = -1;
  en.slot0 = P.T * P.k + kGroup * entry;
  en.M = min(kGroup, P.T - kGroup * entry);
  for (int m = 0; m < kGroup; ++m) en.tok[m] = kGroup * entry + m;
}

// ---------------------------------------------------------------------------
// producer
// ---------------------------------------------------------------------------
// Waits until stage j (issue order) has been released by the consumers.
__device__ __forceinline__ bool wait_released(uint64_t* empty, int NS, int j, const SmallParams& P) {
  return mbar_wait_bounded(&empty[j % NS], (uint32_t)((j / NS) & 1), P.timeout_ns, P.status, kSiteEmpty, j);
}

// The producer is one thread; everything it keeps per stage lives in
// registers or shared memory (no local arrays, no captured locals), since a
// single thread pays the full latency of every dependent access.
template <int L>
__device__ void producer_loop(const SmallParams& P, uint8_t* smem, const SmemPlan& plan) {
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + plan.bars);
  uint64_t* empty = full + P.n_stages;
  Desc* descs = reinterpret_cast<Desc*>(smem + plan.descs);
  Entry* ecache = reinterpret_cast<Entry*>(smem + plan.ecache);
  uint32_t* readybits = reinterpret_cast<uint32_t*>(smem + plan.flags) + 4;  // [8] entries seen published
  constexpr int RB = rec_bytes(L);
  constexpr int XEL = L == 2 ? 2 : 4;  // bytes of one x element
  const int NX = P.n_kt;  // x-record items (one per 512-column slice of x) come first
  const int NR = P.n_rg * P.n_kt;
  const int NSG = P.n_sh * P.n_gu_sh, NSD = P.n_sh * P.n_dt;
  const int NS = P.n_stages;
  // Stage j (in issue order) uses descriptor slot j % NS and `need` bytes of
  // the ring placed right after stage j-1 (or at 0 when the end is reached).
  // Stages [oldest, issued) may still be in flight; their bytes form one arc
  // of the ring that starts at descs[oldest % NS].off and ends at head.
  int issued = 0, oldest = 0, head = 0;
  bool ok = true;
  int n_rent = -1;
  for (int i = 0; i < 8; ++i) readybits[i] = 0u;

  const uint64_t wpol = l2_evict_first_policy();  // weights are read once per launch
  bool st_gu = false, st_dn = false;               // first routed gate/up / down copy stamped
  int t = atomicAdd(&P.sync->queue, 1) - NX;
  while (ok) {
    const int t_next = atomicAdd(&P.sync->queue, 1) - NX;  // claim one ahead: its latency overlaps this tile
    int kind, rgk = 0, rbt, entry = 0, ngroups = 1, nch = 1, nbc, fmt, M, slot0 = 0, n_tiles = 0;
    const Entry* ep = nullptr;
    bool shared_e = false;
    if (t < 0) {
      // an x-record item: the slice of x for all T tokens, no weights
      kind = kXRec;
      rbt = t + NX;
      fmt = MOE_F32;
      nbc = min(kRouterTileChunks, P.n_rc - kRouterTileChunks * rbt);
      M = P.T;
    } else if (t < NR) {
      // a router tile is one stage: the tile's router weights (one contiguous
      // range of the repacked router) and its x slice
      kind = kRouter;
      rgk = (t / P.n_kt) << 16;
      rbt = t % P.n_kt;  // router: index of the 512-column slice
      nch = 1;
      fmt = MOE_F32;
      nbc = min(kRouterTileChunks, P.n_rc - kRouterTileChunks * rbt);  // 128-column chunks in the slice
      M = P.T;
    } else if (t < NR + NSG) {
      kind = kGateUp;
      entry = (t - NR) / P.n_gu_sh;
      rbt = (t - NR) % P.n_gu_sh;
    } else if (t < NR + NSG + NSD) {
      kind = kDown;
      entry = (t - NR - NSG) / P.n_dt;
      rbt = (t - NR - NSG) % P.n_dt;
    } else {
      if (n_rent < 0) {
        if (!wait_flag_geq(&P.sync->routing_ready, P.ready_target, P.timeout_ns, P.status, kSiteRouting, t)) {
          ok = false;
          break;
        }
        fence_proxy_async_global();
        n_rent = __ldcg(&P.sync->n_rent);
        // the routed entries, in one bulk copy (their writers fenced them for
        // the async proxy before the routing flag)
        if (n_rent > 0) {
          uint64_t* ebar = reinterpret_cast<uint64_t*>(smem + plan.ebar);
          const uint32_t eb = (uint32_t)n_rent * (uint32_t)sizeof(Entry);
          mbar_arrive_expect_tx(ebar, eb);
          bulk_g2s(ecache + P.n_sh, P.entries + P.n_sh, eb, ebar);
          if (!mbar_wait_bounded(ebar, 0, P.timeout_ns, P.status, kSiteEntry, -1)) { ok = false; break; }
        }
      }
      const int A = NR + NSG + NSD;
      const int NG = n_rent * P.n_gu, ND = n_rent * P.n_dt;
      if (t < A + NG) {
        kind = kGateUp;
        entry = P.n_sh + (t - A) / P.n_gu;
        rbt = (t - A) % P.n_gu;
      } else if (t < A + NG + ND) {
        kind = kDown;
        entry = P.n_sh + (t - A - NG) / P.n_dt;
        rbt = (t - A - NG) % P.n_dt;
      } else {
        stamp_last(P.stamps, kTsLastIssue);
        break;  // queue exhausted
      }
    }
    const uint8_t* wbase;
    int64_t cbytes;
    int e_id = -1;
    if (kind == kXRec) {
      cbytes = 0;
      wbase = nullptr;
    } else if (kind == kRouter) {
      cbytes = (int64_t)nbc * chunk_bytes(MOE_F32, kRouterCc);
      wbase = P.router + ((int64_t)(rgk >> 16) * P.n_ks * 64 + kRouterTileChunks * 32 * rbt) * kRows * 16;
    } else {
      shared_e = entry < P.n_sh;
      if (shared_e) {
        slot0 = P.T * P.k + kGroup * entry;
        M = min(kGroup, P.T - kGroup * entry);
      } else {
        ep = ecache + entry;
        e_id = ep->e;
        slot0 = ep->slot0;
        M = ep->M;
      }
      fmt = shared_e ? P.sfmt : P.fmt;
      if (kind == kGateUp) {
        ngroups = 2;
        nch = shared_e ? P.sgu_nch : P.gu_nch;
        const int kc = shared_e ? P.sgu_kc : P.gu_kc;
        nbc = kc / 32;
        cbytes = chunk_bytes(fmt, kc);
        wbase = (shared_e ? P.sgu : P.gu + (int64_t)e_id * P.gu_stride) + (int64_t)(2 * rbt) * nch * cbytes;
        n_tiles = shared_e ? P.n_gu_sh : P.n_gu;
      } else {
        ngroups = 4;
        nch = shared_e ? P.sdn_nch : P.dn_nch;
        const int kc = shared_e ? P.sdn_kc : P.dn_kc;
        nbc = kc / 32;
        cbytes = chunk_bytes(fmt, kc);
        wbase = (shared_e ? P.sdn : P.dn + (int64_t)e_id * P.dn_stride) + (int64_t)(4 * rbt) * nch * cbytes;
      }
    }
    const bool xslice = kind == kRouter || kind == kXRec;  // the stage holds a slice of x
    const uint32_t per = xslice ? (uint32_t)(nbc * kRouterCc * XEL) : (uint32_t)(nbc * RB);
    // A group that is one chunk may share its stage with the next groups of
    // the tile (contiguous in memory, same records): fewer, larger stages,
    // as long as two of them fit the ring.
    int gps = 1;
    if (!xslice && nch == 1)
      while (2 * gps <= 4 && ngroups % (2 * gps) == 0 &&
             (int64_t)2 * gps * cbytes + (int64_t)M * per <= (int64_t)(P.ring_bytes / 2))
        gps *= 2;
    const uint32_t wb = (uint32_t)(gps * cbytes);
    const uint32_t resv = wb;
    const int need = (int)((resv + (uint32_t)M * per + 127u) & ~127u);
    // activation sources of this tile at chunk 0, and their step per chunk
    const uint8_t* asrc[kMaxSmallT];
    int64_t astep;
    if (xslice) {
      astep = 0;
#pragma unroll
      for (int m = 0; m < kMaxSmallT; ++m)
        asrc[m] = static_cast<const uint8_t*>(P.x) + ((int64_t)m * P.H + (int64_t)kRouterTileChunks * rbt * kRouterCc) * XEL;
    } else {
      astep = (int64_t)nbc * RB;
#pragma unroll
      for (int m = 0; m < kMaxSmallT; ++m) {
        const int mm = m < kGroup ? m : 0;
        asrc[m] = kind == kGateUp
                      ? P.xrec + (int64_t)(shared_e ? kGroup * entry + mm : ep->tok[mm]) * (P.H / 32) * RB
                      : P.hrec + (int64_t)(slot0 + mm) * (P.Imax / 32) * RB;
      }
    }
    const int4 h3 = make_int4(slot0, P.n_sh + max(n_rent, 0), n_tiles, 0);
    bool dep_ok = xslice;
    if (kind == kGateUp && shared_e) {
      // the shared expert's loads start once the x records exist: in the
      // launch's first microseconds the router tiles, which the routing waits
      // for, get the memory bandwidth
      dep_ok = wait_flag_geq(&P.sync->x_done, P.T * P.n_rc, P.timeout_ns, P.status, kSiteX, t);
      if (dep_ok) fence_proxy_async_global();
      else ok = false;
    }
    const int nstages = ngroups * nch / gps;
    if (e_id >= 0) {
      if (kind == kGateUp && !st_gu) {
        stamp_first(P.stamps, kTsFirstRoutedIssue);
        st_gu = true;
      } else if (kind == kDown && !st_dn) {
        stamp_first(P.stamps, kTsFirstDownIssue);
        st_dn = true;
      }
    }
    for (int q = 0; q < nstages && ok; ++q) {
      const int g = q * gps / nch, c = q * gps - g * nch;
      // ring space: a free slot, then free bytes
      while (ok && issued - oldest >= NS) ok = wait_released(empty, NS, oldest++, P);
      int pos = 0;
      while (ok) {
        pos = head + need <= P.ring_bytes ? head : 0;
        if (oldest == issued) break;
        const int A = descs[oldest & (NS - 1)].off;
        if (A < head ? (pos + need <= A || pos >= head) : (pos >= head && pos + need <= A)) break;
        ok = wait_released(empty, NS, oldest++, P);
      }
      if (!ok) break;
      head = pos + need;
      const int s = issued & (NS - 1);
      const int kch = xslice ? kRouterTileChunks * rbt + c : 0;
      int4* dd = reinterpret_cast<int4*>(descs + s);
      dd[0] = make_int4(kind, c, nch, M);
      dd[1] = make_int4(nbc, fmt, xslice ? rgk | kch : gps, pos);
      dd[2] = make_int4(entry, rbt, g, ngroups);
      dd[3] = h3;
      uint8_t* stage = smem + plan.ring + pos;
      mbar_arrive_expect_tx(&full[s], wb + (uint32_t)M * per);
      if (wb) bulk_g2s_hint(stage, wbase + (int64_t)q * wb, wb, &full[s], wpol);
      if (!dep_ok) {
        if (kind == kGateUp) {
          dep_ok = true;  // routed gate/up: gated by the routing flag (shared: waited above)
        } else if (readybits[entry >> 5] & (1u << (entry & 31))) {
          dep_ok = true;
        } else {
          dep_ok = wait_flag_geq(&P.entry_ready[entry], 1, P.timeout_ns, P.status, kSiteEntry,
                                 entry * 65536 + (t & 0xFFFF));
          if (dep_ok) readybits[entry >> 5] |= 1u << (entry & 31);
        }
        if (dep_ok) fence_proxy_async_global();
        else ok = false;  // the consumers see the status word; the stage is still completed below
      }
      uint8_t* adst = stage + resv;
      const int64_t aoff = (int64_t)c * astep;
#pragma unroll
      for (int m = 0; m < kMaxSmallT; ++m)
        if (m < M) bulk_g2s(adst + m * per, dep_ok ? asrc[m] + aoff : asrc[0], per, &full[s]);
      ++issued;
    }
    t = t_next;
  }
  // end marker (or error): hand the consumers an END descriptor in the next slot
  const int n_data = issued;
  bool have_slot = true;
  while (have_slot && oldest <= issued - NS) have_slot = wait_released(empty, NS, oldest++, P);
  if (have_slot) {
    reinterpret_cast<int4*>(descs + issued % NS)[0] = make_int4(kEnd, 0, 0, 0);
    mbar_arrive(&full[issued % NS]);
  }
  // drain: every bulk copy this CTA issued must have landed before it exits
  for (int j = oldest; j < n_data; ++j)
    mbar_wait_bounded(&full[j % NS], (uint32_t)((j / NS) & 1), P.timeout_ns, P.status, kSiteDrain, j);
}

// ---------------------------------------------------------------------------
// consumer: chunk compute
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t field6(uint32_t w0, uint32_t w1, uint32_t w2, int f) {
  const int p = 6 * f;
  const int wi = p >> 5, sh = p & 31;
  const uint32_t lo = wi == 0 ? w0 : (wi == 1 ? w1 : w2);
  const uint32_t hi = wi == 0 ? w1 : (wi == 1 ? w2 : 0u);
  return __funnelshift_r(lo, hi, sh) & 63u;
}

// Integer dot product of one 32-weight Q8_0 block (codes q0 | q1) with one
// activation record: four independent dp4a chains of four, then the limbs
// combined exactly (L = 2) or in fp32 (L = 4).
template <int L>
__device__ __forceinline__ float q8_block(const uint4 q0, const uint4 q1, const uint8_t* rec) {
  int c[2 * L];
#pragma unroll
  for (int l = 0; l < L; ++l) {
    const uint4 a0 = *reinterpret_cast<const uint4*>(rec + 32 * l);
    const uint4 a1 = *reinterpret_cast<const uint4*>(rec + 32 * l + 16);
    if (l == L - 1) {  // top limb: signed
      c[2 * l] = dp4a_ss(q0.w, a0.w, dp4a_ss(q0.z, a0.z, dp4a_ss(q0.y, a0.y, dp4a_ss(q0.x, a0.x, 0))));
      c[2 * l + 1] = dp4a_ss(q1.w, a1.w, dp4a_ss(q1.z, a1.z, dp4a_ss(q1.y, a1.y, dp4a_ss(q1.x, a1.x, 0))));
    } else {
      c[2 * l] = dp4a_su(q0.w, a0.w, dp4a_su(q0.z, a0.z, dp4a_su(q0.y, a0.y, dp4a_su(q0.x, a0.x, 0))));
      c[2 * l + 1] = dp4a_su(q1.w, a1.w, dp4a_su(q1.z, a1.z, dp4a_su(q1.y, a1.y, dp4a_su(q1.x, a1.x, 0))));
    }
  }
  if constexpr (L == 2) {
    return (float)((c[2] + c[3]) * 256 + (c[0] + c[1]));
  } else {
    return fmaf((float)(c[6] + c[7]), 16777216.f,
                fmaf((float)(c[4] + c[5]), 65536.f, fmaf((float)(c[2] + c[3]), 256.f, (float)(c[0] + c[1]))));
  }
}

// Same for one 32-weight Q4KS sub-block; w[2j] holds codes 8j..8j+3 and
// w[2j+1] codes 8j+4..8j+7, one per byte.
template <int L>
__device__ __forceinline__ float q4_block(const uint32_t (&w)[8], const uint8_t* rec) {
  int c[2 * L];
#pragma unroll
  for (int l = 0; l < L; ++l) {
    const uint4 a0 = *reinterpret_cast<const uint4*>(rec + 32 * l);
    const uint4 a1 = *reinterpret_cast<const uint4*>(rec + 32 * l + 16);
    if (l == L - 1) {
      c[2 * l] = dp4a_us(w[3], a0.w, dp4a_us(w[2], a0.z, dp4a_us(w[1], a0.y, dp4a_us(w[0], a0.x, 0))));
      c[2 * l + 1] = dp4a_us(w[7], a1.w, dp4a_us(w[6], a1.z, dp4a_us(w[5], a1.y, dp4a_us(w[4], a1.x, 0))));
    } else {
      c[2 * l] = dp4a_uu(w[3], a0.w, dp4a_uu(w[2], a0.z, dp4a_uu(w[1], a0.y, dp4a_uu(w[0], a0.x, 0))));
      c[2 * l + 1] = dp4a_uu(w[7], a1.w, dp4a_uu(w[6], a1.z, dp4a_uu(w[5], a1.y, dp4a_uu(w[4], a1.x, 0))));
    }
  }
  if constexpr (L == 2) {
    return (float)((c[2] + c[3]) * 256 + (c[0] + c[1]));
  } else {
    return fmaf((float)(c[6] + c[7]), 16777216.f,
                fmaf((float)(c[4] + c[5]), 65536.f, fmaf((float)(c[2] + c[3]), 256.f, (float)(c[0] + c[1]))));
  }
}

__device__ __forceinline__ void q4_unpack(const uint4 qv, uint32_t (&w)[8]) {
  w[0] = qv.x & 0x0F0F0F0Fu; w[1] = (qv.x >> 4) & 0x0F0F0F0Fu;
  w[2] = qv.y & 0x0F0F0F0Fu; w[3] = (qv.y >> 4) & 0x0F0F0F0Fu;
  w[4] = qv.z & 0x0F0F0F0Fu; w[5] = (qv.z >> 4) & 0x0F0F0F0Fu;
  w[6] = qv.w & 0x0F0F0F0Fu; w[7] = (qv.w >> 4) & 0x0F0F0F0Fu;
}

// a = d * sc[s], b = dmin * m[s] of sub-block s from a 16-byte superblock header
__device__ __forceinline__ void q4_scales(const uint4 hd, int s, float& a, float& b) {
  const float dd = __half2float(__ushort_as_half((unsigned short)(hd.x & 0xFFFFu)));
  const float dmin = __half2float(__ushort_as_half((unsigned short)(hd.x >> 16)));
  a = dd * (float)field6(hd.y, hd.z, hd.w, s);
  b = dmin * (float)field6(hd.y, hd.z, hd.w, 8 + s);
}

// One chunk.  Lane l owns row l of the chunk; warp w owns blocks w, w + 8,
// ... (a warp load of one block's 16-byte pieces covers the 32 rows in 512
// contiguous bytes; the block's activation records are a broadcast read, one
// per warp).  acc[m] collects this warp's share of the lane's row against
// vector m; the 8 warps' shares are summed by the epilogue warp.
template <int L, int M>
__device__ __forceinline__ void gemv_chunk_m(const uint8_t* stage, const uint8_t* A, int nbc, int fmt,
                                             float (&acc)[kGroup]) {
  constexpr int RB = rec_bytes(L);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (fmt == MOE_Q8_0) {
    const __half* sc = reinterpret_cast<const __half*>(stage + nbc * 1024);
#pragma unroll 2
    for (int b = warp; b < nbc; b += kBlocksPerStep) {
      const uint4 q0 = *reinterpret_cast<const uint4*>(stage + ((int64_t)(b * 2 + 0) * kRows + lane) * 16);
      const uint4 q1 = *reinterpret_cast<const uint4*>(stage + ((int64_t)(b * 2 + 1) * kRows + lane) * 16);
      const float dq = __half2float(sc[b * kRows + lane]);
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const uint8_t* rec = A + (m * nbc + b) * RB;
        const float asc = *reinterpret_cast<const float*>(rec + 32 * L);
        acc[m] = fmaf(dq * asc, q8_block<L>(q0, q1, rec), acc[m]);
      }
    }
  } else {  // MOE_Q4KS
    const uint8_t* hdr = stage + nbc * 512;
#pragma unroll 2
    for (int b = warp; b < nbc; b += kBlocksPerStep) {
      const uint4 qv = *reinterpret_cast<const uint4*>(stage + ((int64_t)b * kRows + lane) * 16);
      const uint4 hd = *reinterpret_cast<const uint4*>(hdr + ((b >> 3) * kRows + lane) * 16);
      float sa, sb;
      q4_scales(hd, b & 7, sa, sb);
      uint32_t w[8];
      q4_unpack(qv, w);
#pragma unroll
      for (int m = 0; m < M; ++m) {
        const uint8_t* rec = A + (m * nbc + b) * RB;
        const float asc = reinterpret_cast<const float*>(rec + 32 * L)[0];
        const float sx = reinterpret_cast<const float*>(rec + 32 * L)[1];
        acc[m] = fmaf(sa * asc, q4_block<L>(w, rec), fmaf(-sb, sx, acc[m]));
      }
    }
  }
}

// The token count of a stage as a compile-time constant, so the loops over
// tokens unroll without predicates (a runtime bound there keeps the loads of
// different tokens from being scheduled together).
template <int L>
__device__ __forceinline__ void gemv_chunk(const uint8_t* stage, const uint8_t* A, int nbc, int fmt, int M,
                                           float (&acc)[kGroup]) {
  switch (M) {
    case 1: gemv_chunk_m<L, 1>(stage, A, nbc, fmt, acc); break;
    case 2: gemv_chunk_m<L, 2>(stage, A, nbc, fmt, acc); break;
    case 3: gemv_chunk_m<L, 3>(stage, A, nbc, fmt, acc); break;
    default: gemv_chunk_m<L, kGroup>(stage, A, nbc, fmt, acc); break;
  }
}

// ---------------------------------------------------------------------------
// consumer: routing (last router tile)
// ---------------------------------------------------------------------------
// fp32 -> unsigned key with the same order (no NaNs; -0 is mapped to +0 first).
__device__ __forceinline__ uint32_t order_key(float f) {
  const uint32_t u = __float_as_uint(f + 0.0f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Largest of N values by a pairwise tree (depth log2 N).
template <int N>
__device__ __forceinline__ uint64_t tree_max(const uint64_t (&c)[N]) {
  uint64_t t[N];
#pragma unroll
  for (int i = 0; i < N; ++i) t[i] = c[i];
#pragma unroll
  for (int w = 1; w < N; w <<= 1)
#pragma unroll
    for (int i = 0; i + w < N; i += 2 * w) t[i] = t[i] > t[i + w] ? t[i] : t[i + w];
  return t[0];
}

// The k largest of row[0..E) by (value desc, index asc), one warp.  Lane l
// holds experts l, l + 32, ... (NPER of them) in registers as 64-bit
// composites (order-preserving key of the value, then the complemented index,
// so a larger composite is a larger value or, on equal values, a lower
// index; 0 = none) and keeps its largest.  Each round takes the exact maximum
// key over the lanes (a warp max); if several lanes hold it, the lowest
// expert index among them wins (a second warp min, only then).  The winning
// lane writes the slot, clears that expert and takes the tree maximum of what
// it has left.  NaN counts as -inf.  Writes ids and values in slot order.
template <int NPER>
__device__ __forceinline__ void topk_token(const float* row, int E, int k, int* ids, float* vals_out) {
  const int lane = threadIdx.x & 31;
  uint64_t c[NPER];
#pragma unroll
  for (int i = 0; i < NPER; ++i) {
    const int e = lane + 32 * i;
    const float x = e < E ? row[e] : 0.f;
    c[i] = e < E ? ((uint64_t)order_key(x == x ? x : -INFINITY) << 32) | (uint64_t)(~(uint32_t)e) : 0ull;
  }
  uint64_t best = tree_max(c);
#pragma unroll 1
  for (int j = 0; j < k; ++j) {
    const uint32_t key = (uint32_t)(best >> 32);
    const uint32_t m = __reduce_max_sync(0xffffffffu, key);
    const uint32_t holders = __ballot_sync(0xffffffffu, best != 0ull && key == m);
    int wl = __ffs(holders) - 1;
    if (holders & (holders - 1u))
      wl = (int)(__reduce_min_sync(0xffffffffu, (holders >> lane) & 1u ? ~(uint32_t)best : 0x7fffffffu) & 31u);
    if (lane == wl) {
      const uint32_t wi = ~(uint32_t)best;
      ids[j] = (int)wi;
      vals_out[j] = key_value(m);
      const int slot = (int)(wi >> 5);
#pragma unroll
      for (int i = 0; i < NPER; ++i)
        if (i == slot) c[i] = 0ull;
      best = tree_max(c);
    }
  }
}

// Scratch of finalize_routing in the misc region (bytes, see finalize_misc_bytes).
struct FinLayout {
  int lg, sid, sl, sg, sperm, spos, slt, srank, sent, end;
};
__host__ __device__ inline FinLayout fin_layout(int T, int E, int k) {
  const int t4 = (T * k + 3) & ~3;
  FinLayout f;
  f.lg = 0;
  f.sid = ((T * E * 4 + 15) & ~15);
  f.sl = f.sid + 4 * t4;
  f.sg = f.sl + 4 * t4;
  f.sperm = f.sg + 4 * t4;
  f.spos = f.sperm + 4 * t4;
  f.slt = f.spos + 4 * t4;
  f.srank = f.slt + 4 * t4;
  f.sent = f.srank + 4 * t4;
  f.end = f.sent + 4 * t4;
  return f;
}
int finalize_misc_bytes(int T, int E, int k) { return fin_layout(T, E, k).end + 16; }

// Runs on the consumer threads of the CTA that finished the last router
// tile: logits, top-k and gates, then the permutation and the routed work
// entries.  The entries and their count are published first (routing_ready);
// ids, gates, offsets, perm and pos follow (routing_aux), since only the
// combine and moe_get_routing read them.  A layer that holds only the routed
// experts [e0, e0 + n_e) (one shard of an expert-parallel split) routes over
// all E experts but makes entries for its own only; their expert field is the
// local index e - e0.
//
// With Tk = T * k <= 128 pairs, pair p finds its place by counting: lt = the
// pairs of lower experts, rank = the earlier pairs of its own expert, so its
// slot is lt + rank (experts ascending, tokens ascending within an expert).
// The first pair of an expert owns that expert's entries: its entry index is
// the number of entries of all lower experts.
__device__ void finalize_routing(const SmallParams& P, uint8_t* misc, int* pend) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NT = kConsumerWarps * 32;
  const int T = P.T, E = P.E, k = P.k, Tk = P.T * P.k;
  const FinLayout f = fin_layout(T, E, k);
  float* lg = reinterpret_cast<float*>(misc + f.lg);    // [T*E]
  int* sid = reinterpret_cast<int*>(misc + f.sid);      // [Tk]
  float* sl = reinterpret_cast<float*>(misc + f.sl);    // [Tk]
  float* sg = reinterpret_cast<float*>(misc + f.sg);    // [Tk]
  int* sperm = reinterpret_cast<int*>(misc + f.sperm);  // [Tk]
  int* spos = reinterpret_cast<int*>(misc + f.spos);    // [Tk]
  int* slt = reinterpret_cast<int*>(misc + f.slt);      // [Tk] pairs of lower experts
  int* srank = reinterpret_cast<int*>(misc + f.srank);  // [Tk] earlier pairs of the same expert
  int* sent = reinterpret_cast<int*>(misc + f.sent);    // [Tk] entries owned (first pair of an expert)

  // (the router counter was taken with acquire semantics)
  // logits: thread i converts the fixed-point sums of experts e = i, i + 256
  // (all loads in flight before the conversions), then any further experts
  {
    const int nq = P.Tp / 2;  // 16-byte pairs per expert (Tp <= 8)
    const longlong2* lp = reinterpret_cast<const longlong2*>(P.lfx);
    auto put = [&](int e, const longlong2* a) {
      const float bias = P.router_b ? P.router_b[e] : 0.f;
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q < nq) {
          // one rounding to fp32, then an exact power-of-two scale
          if (2 * q < T) lg[(2 * q) * E + e] = __ll2float_rn(a[q].x) * 0x1p-32f + bias;
          if (2 * q + 1 < T) lg[(2 * q + 1) * E + e] = __ll2float_rn(a[q].y) * 0x1p-32f + bias;
        }
    };
    longlong2 a[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (tid + u * NT < E && q < nq) a[u][q] = __ldcg(lp + (int64_t)(tid + u * NT) * nq + q);
#pragma unroll
    for (int u = 0; u < 2; ++u)
      if (tid + u * NT < E) put(tid + u * NT, a[u]);
#pragma unroll 1
    for (int e = tid + 2 * NT; e < E; e += NT) {  // E > 512
      longlong2 c[4];
#pragma unroll
      for (int q = 0; q < 4; ++q)
        if (q < nq) c[q] = __ldcg(lp + (int64_t)e * nq + q);
      put(e, c);
    }
  }
  consumer_sync();

  // top-k and gates per token (one warp per token)
  const int nper = (E + 31) / 32;
#pragma unroll 1
  for (int t = warp; t < T; t += kConsumerWarps) {
    if (nper <= 4) topk_token<4>(lg + t * E, E, k, sid + t * k, sl + t * k);
    else if (nper <= 8) topk_token<8>(lg + t * E, E, k, sid + t * k, sl + t * k);
    else if (nper <= 12) topk_token<12>(lg + t * E, E, k, sid + t * k, sl + t * k);
    else if (nper <= 16) topk_token<16>(lg + t * E, E, k, sid + t * k, sl + t * k);
    else topk_token<kMaxE / 32>(lg + t * E, E, k, sid + t * k, sl + t * k);
    __syncwarp();
    // gates: softmax over the k selected logits (lane j: slot j), the sum by
    // a fixed shuffle tree
    const float l0 = sl[t * k];
    const float ex = lane < k ? expf(sl[t * k + lane] - l0) : 0.f;
    float sum = ex;
#pragma unroll
    for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
    if (lane < k) sg[t * k + lane] = ex / sum;
  }
  consumer_sync();

  // slot of each pair (experts ascending, tokens ascending within an
  // expert) and the routed entries (up to kGroup consecutive slots of one
  // expert each, in slot order)
  int n_rent = 0;
  if (Tk <= 32) {
    // one warp, lane p = pair p.  lt = pairs of lower experts, by a radix
    // over the bits of the expert index (lanes past Tk get expert 1024,
    // above every real one); eq ends as the lanes with my expert.
    if (warp == 0) {
      const bool act = lane < Tk;
      const int ekey = act ? sid[lane] : 1024;
      int lt = 0;
      uint32_t eq = 0xffffffffu;
#pragma unroll
      for (int b = 10; b >= 0; --b) {
        const bool bit = (ekey >> b) & 1;
        const uint32_t ones = __ballot_sync(0xffffffffu, bit);
        if (bit) lt += __popc(eq & ~ones);
        eq &= bit ? ones : ~ones;
      }
      const uint32_t below = (1u << lane) - 1u;
      const int rank = __popc(eq & below), cnt = __popc(eq);
      if (act) {
        sperm[lt + rank] = lane;
        spos[lane] = lt + rank;
      }
      __syncwarp();
      // slot view: lane i holds the pair at slot i
      const int q = act ? sperm[lane] : 0;
      const int e_i = __shfl_sync(0xffffffffu, ekey, q);
      const int r_i = __shfl_sync(0xffffffffu, rank, q);
      const int c_i = __shfl_sync(0xffffffffu, cnt, q);
      const int tok = q / k;
      const bool own = e_i >= P.e0 && e_i < P.e0 + P.n_e;
      const uint32_t starts = __ballot_sync(0xffffffffu, act && own && r_i % kGroup == 0);
      int tk[kGroup];
      tk[0] = tok;
#pragma unroll
      for (int m = 1; m < kGroup; ++m) tk[m] = __shfl_down_sync(0xffffffffu, tok, m);
      if ((starts >> lane) & 1u) {
        const int M = min(kGroup, c_i - r_i);
        int4* dst = reinterpret_cast<int4*>(P.entries + P.n_sh + __popc(starts & below));
        dst[0] = make_int4(e_i - P.e0, lane, M, tk[0]);
        dst[1] = make_int4(M > 1 ? tk[1] : 0, M > 2 ? tk[2] : 0, M > 3 ? tk[3] : 0, 0);
        fence_proxy_async_global();  // the producers fetch the entries with a bulk copy
      }
      n_rent = __popc(starts);
    }
  } else {
    // general case: pair p counts over all pairs
    const int4* sid4 = reinterpret_cast<const int4*>(sid);
    const int4* sent4 = reinterpret_cast<const int4*>(sent);
    const int nq4 = (Tk + 3) / 4;
    if (tid < Tk) {
      const int p = tid, e = sid[p];
      int lt = 0, rank = 0, c = 0;
#pragma unroll 4
      for (int q4 = 0; q4 < nq4; ++q4) {
        const int4 v = sid4[q4];
        const int ev[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int q = 4 * q4 + u;
          if (q < Tk) {
            lt += ev[u] < e;
            rank += (ev[u] == e) & (q < p);
            c += ev[u] == e;
          }
        }
      }
      const int slot = lt + rank;
      sperm[slot] = p;
      spos[p] = slot;
      slt[p] = lt;
      srank[p] = rank;
      sent[p] = rank == 0 && e >= P.e0 && e < P.e0 + P.n_e ? (c + kGroup - 1) / kGroup : 0;
    }
    consumer_sync();
    // entries: the first pair of each expert writes them (tokens from the
    // permutation); its entry index is the entry count of the lower experts
    if (tid < Tk && srank[tid] == 0) {
      const int e = sid[tid], lt = slt[tid], ne = sent[tid];
      int w0 = 0, c = 0;
#pragma unroll 4
      for (int q4 = 0; q4 < nq4; ++q4) {
        const int4 v = sid4[q4], n = sent4[q4];
        const int ev[4] = {v.x, v.y, v.z, v.w}, nv[4] = {n.x, n.y, n.z, n.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (4 * q4 + u < Tk) {
            w0 += ev[u] < e ? nv[u] : 0;
            c += ev[u] == e;
          }
      }
#pragma unroll 1
      for (int g = 0; g < ne; ++g) {
        const int slot0 = lt + g * kGroup, M = min(kGroup, c - g * kGroup);
        int tok[kGroup];
#pragma unroll
        for (int m = 0; m < kGroup; ++m) tok[m] = m < M ? sperm[slot0 + m] / k : 0;
        int4* dst = reinterpret_cast<int4*>(P.entries + P.n_sh + w0 + g);
        dst[0] = make_int4(e - P.e0, slot0, M, tok[0]);
        dst[1] = make_int4(tok[1], tok[2], tok[3], 0);
      }
      fence_proxy_async_global();  // the producers fetch the entries with a bulk copy
    }
    if (tid == 0) {
#pragma unroll 4
      for (int q4 = 0; q4 < nq4; ++q4) {
        const int4 n = sent4[q4];
        const int nv[4] = {n.x, n.y, n.z, n.w};
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (4 * q4 + u < Tk) n_rent += nv[u];
      }
    }
  }
  consumer_sync();
  // the barrier orders every thread's entry writes before thread 0's release
  int* nrent_s = reinterpret_cast<int*>(misc + f.end);
  if (tid == 0) {
    P.sync->n_rent = n_rent;
    st_release(&P.sync->routing_ready, 1);
    stamp_last(P.stamps, kTsRoutingReady);
    *nrent_s = n_rent;
  }
  consumer_sync();
  // One arrival of the routing on every 128-row block of z: a block is
  // complete after n_sh + n_rent down tiles and this arrival, and whoever
  // arrives last combines it.  A shared down tile that finishes before the
  // routing is known can therefore never be taken for the last one, and a
  // layer with no down work for this batch (a shard none of whose experts
  // was chosen, with no shared expert) still gets y from the combine.
  {
    const int last = P.n_sh + *nrent_s;
    for (int b = tid; b < P.n_dt; b += NT)
      if (atom_add_acq_rel(&P.d_cnt[b], 1) == last) pend[1 + atomicAdd(&pend[0], 1)] = b;
  }
  // what only the combine and moe_get_routing read
  if (tid < Tk) {
    P.ids[tid] = sid[tid];
    P.gates[tid] = sg[tid];
    P.perm[tid] = sperm[tid];
    P.pos[tid] = spos[tid];
  }
#pragma unroll 1
  for (int e = tid; e <= E; e += NT) {
    int o = 0;
#pragma unroll 4
    for (int q = 0; q < Tk; ++q) o += sid[q] < e;
    P.offsets[e] = o;
  }
  consumer_sync();
  if (tid == 0) st_release(&P.sync->routing_aux, 1);
}

// Router tile dot products: lane = expert row, warp w takes float4 columns
// w, w + 8, ... of the slice; T tokens (compile time), four independent
// accumulators per token (one per float4 component).
template <int L, int T>
__device__ __forceinline__ void router_dot(const float4* wst, const uint8_t* xs, int cols, float (&racc)[kMaxSmallT]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float ra[T][4];
#pragma unroll
  for (int t = 0; t < T; ++t)
#pragma unroll
    for (int c = 0; c < 4; ++c) ra[t][c] = 0.f;
  const int ncol4 = cols / 4;
#pragma unroll 4
  for (int i = 0; i < 16; ++i) {
    const int k4 = warp + kConsumerWarps * i;
    if (k4 < ncol4) {
      const float4 w = wst[k4 * 32 + lane];
#pragma unroll
      for (int t = 0; t < T; ++t) {
        float4 xv;
        if constexpr (L == 2) {
          const uint2 raw = *reinterpret_cast<const uint2*>(xs + (t * cols + k4 * 4) * 2);
          xv = make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u),
                           __uint_as_float(raw.y << 16), __uint_as_float(raw.y & 0xFFFF0000u));
        } else {
          xv = *reinterpret_cast<const float4*>(xs + (t * cols + k4 * 4) * 4);
        }
        ra[t][0] = fmaf(w.x, xv.x, ra[t][0]);
        ra[t][1] = fmaf(w.y, xv.y, ra[t][1]);
        ra[t][2] = fmaf(w.z, xv.z, ra[t][2]);
        ra[t][3] = fmaf(w.w, xv.w, ra[t][3]);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kMaxSmallT; ++t) racc[t] = t < T ? (ra[t][0] + ra[t][1]) + (ra[t][2] + ra[t][3]) : 0.f;
}

// ---------------------------------------------------------------------------
// consumers
// ---------------------------------------------------------------------------
template <int L>
__device__ void consumer_loop(const SmallParams& P, uint8_t* smem, const SmemPlan& plan) {
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + plan.bars);
  uint64_t* empty = full + P.n_stages;
  uint64_t* rfull = reinterpret_cast<uint64_t*>(smem + plan.rbars);
  uint64_t* rempty = rfull + kRedSlots;
  const Desc* descs = reinterpret_cast<const Desc*>(smem + plan.descs);
  Desc* metas = reinterpret_cast<Desc*>(smem + plan.metas);
  float* rred = reinterpret_cast<float*>(smem + plan.rred);  // [8 warps][8 tokens][32]
  float* red = reinterpret_cast<float*>(smem + plan.red);    // [slot][8 warps][4][32]
  uint8_t* misc = smem + plan.misc;
  int* flags = reinterpret_cast<int*>(smem + plan.flags);
  constexpr int RB = rec_bytes(L);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int T = P.T;
  int s = 0, rs = 0;
  uint32_t ph = 0, rph = 0;
  float acc[kGroup];
  float racc[kMaxSmallT];
  bool st_routed = false;  // (thread 0) first routed gate/up stage stamped

  while (true) {
    if (!mbar_wait_bounded(&full[s], ph, P.timeout_ns, P.status, kSiteFull, s)) break;
    Desc d;  // consumers need only the first 32 bytes; thread 0 copies the rest for the epilogue
    {
      const int4* src = reinterpret_cast<const int4*>(descs + s);
      const int4 h0 = src[0], h1 = src[1];
      d.kind = h0.x; d.chunk = h0.y; d.nch = h0.z; d.M = h0.w;
      d.nbc = h1.x; d.fmt = h1.y; d.rgks = h1.z; d.off = h1.w;
      if (tid == 0) {
        const int4 h2 = src[2], h3 = src[3];
        d.entry = h2.x; d.rbt = h2.y; d.group = h2.z; d.ngroups = h2.w;
        d.slot0 = h3.x; d.n_ent = h3.y; d.n_tiles_entry = h3.z; d.pad = h3.w;
      }
    }
    if (d.kind == kEnd) {
      // pass the end marker on to the epilogue warp
      if (mbar_wait_bounded(&rempty[rs], rph ^ 1u, P.timeout_ns, P.status, kSiteRedEmpty, rs)) {
        if (tid == 0) metas[rs] = d;
        __syncwarp();
        if (lane == 0) mbar_arrive(&rfull[rs]);
      }
      break;
    }
    const uint8_t* stage = smem + plan.ring + d.off;
    const int d_rg = d.rgks >> 16, d_ks = d.rgks & 0xFFFF;  // router tiles

    if (d.kind == kXRec) {
      // x slice ([T][cols] in the stage) -> activation records, one 32-column
      // block per thread; the proxy fence makes them visible to the bulk
      // copies that read them after x_done
      const int kt = d_ks / kRouterTileChunks, cols = d.nbc * kRouterCc, nb = cols / 32;
      constexpr int XEL = L == 2 ? 2 : 4;
      if (tid < T * nb) {
        const int t = tid / nb, b = tid - (tid / nb) * nb;
        write_record_lane<L>(stage + (t * cols + b * 32) * XEL,
                             P.xrec + ((int64_t)t * (P.H / 32) + kt * (kRouterTileChunks * kRouterCc / 32) + b) * RB);
        fence_proxy_async_global();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
      consumer_sync();  // orders every thread's record writes before thread 0's release
      if (tid == 0 && atom_add_acq_rel(&P.sync->x_done, T * d.nbc) + T * d.nbc == T * P.n_rc)
        stamp_last(P.stamps, kTsXDone);
    } else if (d.kind == kRouter) {
      // One router tile: 32 experts (lane = expert row) x a slice of ncc
      // 128-column chunks.  The stage holds the tile's router weights
      // ([cols/4][32 rows][4]) and then the slice of x ([T][cols]).
      const int ncc = d.nbc, cols = ncc * kRouterCc;
      const float4* wst = reinterpret_cast<const float4*>(stage);
      const uint8_t* xs = stage + cols * kRows * 4;
      switch (T) {
        case 1: router_dot<L, 1>(wst, xs, cols, racc); break;
        case 2: router_dot<L, 2>(wst, xs, cols, racc); break;
        case 3: router_dot<L, 3>(wst, xs, cols, racc); break;
        case 4: router_dot<L, 4>(wst, xs, cols, racc); break;
        case 5: router_dot<L, 5>(wst, xs, cols, racc); break;
        case 6: router_dot<L, 6>(wst, xs, cols, racc); break;
        case 7: router_dot<L, 7>(wst, xs, cols, racc); break;
        default: router_dot<L, 8>(wst, xs, cols, racc); break;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);
#pragma unroll
      for (int t = 0; t < kMaxSmallT; ++t)
        if (t < T) rred[(warp * kMaxSmallT + t) * 32 + lane] = racc[t];
      consumer_sync();
      if (tid < T * 32) {
        // this slice's share of logit (t, expert 32 rg + r), added as an
        // exact integer multiple of 2^-32: the total does not depend on the
        // order in which the slices arrive
        const int t = tid >> 5, r = tid & 31;
        float v = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) v += rred[(w * kMaxSmallT + t) * 32 + r];
        atomicAdd(reinterpret_cast<unsigned long long*>(P.lfx) + (int64_t)(d_rg * 32 + r) * P.Tp + t,
                  (unsigned long long)__float2ll_rn(v * 4294967296.f));
      }
      // the barrier orders every thread's additions before thread 0's
      // release (acquire-release) count
      consumer_sync();
      if (tid == 0) {
        const int old = atom_add_acq_rel(&P.sync->router_done, 1);
        flags[0] = (old == P.n_rg * P.n_kt - 1);
      }
      consumer_sync();
      if (flags[0]) {
        if (tid == 0) stamp_last(P.stamps, kTsRouterDone);
        finalize_routing(P, misc, reinterpret_cast<int*>(smem + plan.pend));
      }
      consumer_sync();
    } else {
      // gate/up or down: one chunk of a group, or gps whole groups of one
      // chunk each (their weights back to back, then the shared records)
      const int gps = d.rgks;
      const int cb = (int)chunk_bytes(d.fmt, d.nbc * 32);
      if (tid == 0 && !st_routed && d.kind == kGateUp && d.entry >= P.n_sh) {
        stamp_first(P.stamps, kTsFirstRoutedCompute);
        st_routed = true;
      }
      const uint8_t* recs = stage + gps * cb;
      bool failed = false;
      for (int j = 0; j < gps; ++j) {
        if (d.chunk == 0) {
#pragma unroll
          for (int m = 0; m < kGroup; ++m) acc[m] = 0.f;
        }
        gemv_chunk<L>(stage + j * cb, recs, d.nbc, d.fmt, d.M, acc);
        if (j == gps - 1) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&empty[s]);
        }
        if (d.chunk == d.nch - 1) {
          // a 32-row group is complete: hand this warp's share of every row to
          // the epilogue warp (the descriptor is copied before the stage is
          // released, since the producer reuses it)
          if (!mbar_wait_bounded(&rempty[rs], rph ^ 1u, P.timeout_ns, P.status, kSiteRedEmpty, rs)) {
            failed = true;
            break;
          }
          float4* slot = reinterpret_cast<float4*>(red + rs * (kRedSlotBytes / 4));  // [warp][row][token]
          slot[warp * kRows + lane] = make_float4(acc[0], acc[1], acc[2], acc[3]);
          if (tid == 0) {
            Desc dj = d;
            dj.group = d.group + j;
            metas[rs] = dj;
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(&rfull[rs]);
          if (++rs == kRedSlots) { rs = 0; rph ^= 1u; }
        }
      }
      if (failed) break;
    }
    if (++s == P.n_stages) { s = 0; ph ^= 1u; }
  }
}

// ---------------------------------------------------------------------------
// epilogue warp
// ---------------------------------------------------------------------------
template <int L>
__device__ void epilogue_loop(const SmallParams& P, uint8_t* smem, const SmemPlan& plan) {
  uint64_t* rfull = reinterpret_cast<uint64_t*>(smem + plan.rbars);
  uint64_t* rempty = rfull + kRedSlots;
  const Desc* metas = reinterpret_cast<const Desc*>(smem + plan.metas);
  const float* red = reinterpret_cast<const float*>(smem + plan.red);
  constexpr int RB = rec_bytes(L);
  const int lane = threadIdx.x & 31;
  int rs = 0;
  uint32_t rph = 0;
  float keep[kGroup] = {0.f, 0.f, 0.f, 0.f};
  while (true) {
    if (!mbar_wait_bounded(&rfull[rs], rph, P.timeout_ns, P.status, kSiteRedFull, rs)) break;
    const Desc d = metas[rs];
    if (d.kind == kEnd) break;
    // row = lane: sum the consumer warps' shares in warp order
    const float4* slot = reinterpret_cast<const float4*>(red + rs * (kRedSlotBytes / 4));
    float v[kGroup] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int w = 0; w < kConsumerWarps; ++w) {
      const float4 x = slot[w * kRows + lane];
      v[0] += x.x; v[1] += x.y; v[2] += x.z; v[3] += x.w;
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&rempty[rs]);
    if (++rs == kRedSlots) { rs = 0; rph ^= 1u; }

    if (d.kind == kGateUp) {
      // lanes 0-15: gate rows, lanes 16-31: up rows of outputs 32*rbt + 16*group + (0..15)
#pragma unroll
      for (int m = 0; m < kGroup; ++m) {
        const float u = __shfl_down_sync(0xffffffffu, v[m], 16);
        const float hv = v[m] / (1.f + expf(-v[m])) * u;  // meaningful on lanes 0-15
        if (d.group == 0) {
          keep[m] = hv;
        } else {
          const float hi = __shfl_up_sync(0xffffffffu, hv, 16);
          const float vec = lane < 16 ? keep[m] : hi;
          if (m < d.M)
            write_record<L>(vec, P.hrec + ((int64_t)(d.slot0 + m) * (P.Imax / 32) + d.rbt) * RB);
        }
      }
      if (d.group == d.ngroups - 1) {
        // the records are read by bulk copies; __syncwarp orders the lanes'
        // writes before lane 0's acquire-release count, whose release covers
        // them and, for the last tile, those of the tiles counted before it
        fence_proxy_async_global();
        __syncwarp();
        if (lane == 0 && atom_add_acq_rel(&P.gu_cnt[d.entry], 1) == d.n_tiles_entry - 1) {
          st_release(&P.entry_ready[d.entry], 1);
          stamp_last(P.stamps, d.entry < P.n_sh ? kTsSharedGateUp : kTsLastGateUp);
        }
      }
    } else {  // kDown
      const int row = d.rbt * 128 + d.group * 32 + lane;
      for (int m = 0; m < d.M; ++m) P.z[(int64_t)(d.slot0 + m) * P.H + row] = v[m];
      if (d.group == d.ngroups - 1) {
        __syncwarp();  // orders the lanes' z writes before lane 0's release
        if (lane == 0) {
          // the block is complete after every down tile (n_sh + n_rent) and
          // the routing's own arrival; n_rent is visible whenever the routing
          // has arrived, and before that no tile can be the last one
          const int old = atom_add_acq_rel(&P.d_cnt[d.rbt], 1);
          if (old == P.n_sh + ld_acquire(&P.sync->n_rent)) {
            stamp_last(P.stamps, kTsLastDownDone);
            // this CTA combines the block when it leaves (with all its threads)
            int* pend = reinterpret_cast<int*>(smem + plan.pend);
            pend[1 + atomicAdd(&pend[0], 1)] = d.rbt;
          }
        }
      }
    }
  }
}

// y rows of the 128-row blocks this CTA completed last, in slot order:
// y[t] = sum_{j<k} g[t,j] z[pos[t,j]] + z_shared[t], all threads of the CTA.
template <int L>
__device__ void combine_blocks(const SmallParams& P, uint8_t* smem, const SmemPlan& plan, const int* pend) {
  float* sg = reinterpret_cast<float*>(smem + plan.escr);                       // [T*k] gates
  int* sp = reinterpret_cast<int*>(smem + plan.escr + kMaxSmallT * kMaxTopK * 4);  // [T*k] slots
  const int T = P.T, k = P.k;
  int* flags = reinterpret_cast<int*>(smem + plan.flags);
  __threadfence();
  if (threadIdx.x == 0)  // set right after the routing; long done by now
    flags[2] = wait_flag_geq(&P.sync->routing_aux, 1, P.timeout_ns, P.status, kSiteRouting, -1);
  __syncthreads();
  if (!flags[2]) return;
  for (int q = threadIdx.x; q < T * k; q += blockDim.x) {
    const int e = __ldcg(&P.ids[q]);
    sg[q] = __ldcg(&P.gates[q]);
    sp[q] = e >= P.e0 && e < P.e0 + P.n_e ? __ldcg(&P.pos[q]) : -1;  // -1: another shard's expert
  }
  __syncthreads();
  const int n = pend[0];
  for (int o = threadIdx.x; o < n * 128 * T; o += blockDim.x) {
    const int b = o / (128 * T), rem = o % (128 * T), t = rem / 128;
    const int r = pend[1 + b] * 128 + rem % 128;
    float zv[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k) zv[j] = sp[t * k + j] >= 0 ? __ldcg(&P.z[(int64_t)sp[t * k + j] * P.H + r]) : 0.f;
    const float zs = P.n_sh > 0 ? __ldcg(&P.z[(int64_t)(T * k + t) * P.H + r]) : 0.f;
    float acc = 0.f;
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k && sp[t * k + j] >= 0) acc = fmaf(sg[t * k + j], zv[j], acc);
    acc += zs;
    if (P.residual) {
      if constexpr (L == 2) acc += __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(P.x)[(int64_t)t * P.H + r]);
      else acc += reinterpret_cast<const float*>(P.x)[(int64_t)t * P.H + r];
    }
    if constexpr (L == 2) reinterpret_cast<__nv_bfloat16*>(P.y)[(int64_t)t * P.H + r] = __float2bfloat16_rn(acc);
    else reinterpret_cast<float*>(P.y)[(int64_t)t * P.H + r] = acc;
  }
}

template <int L>
__global__ void __launch_bounds__(kThreads, 1) moe_small_t_kernel(const __grid_constant__ SmallParams P) {
  extern __shared__ __align__(128) uint8_t smem[];
  const SmemPlan plan = smem_plan(P.n_stages, P.ring_bytes, P.misc_bytes, P.w_max);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + plan.bars);
  uint64_t* empty = full + P.n_stages;
  uint64_t* rfull = reinterpret_cast<uint64_t*>(smem + plan.rbars);
  uint64_t* rempty = rfull + kRedSlots;
  int* flags = reinterpret_cast<int*>(smem + plan.flags);
  int* pend = reinterpret_cast<int*>(smem + plan.pend);
  // The next launch in the stream may start as this one's CTAs leave; until
  // griddep_wait it touches nothing this launch (or an earlier one) writes.
  griddep_launch_dependents();
  const uint64_t t_entry = globaltimer_ns();
  if (threadIdx.x == 0) {
    // constant data only: warm L2 with one router tile's weights (tile = CTA)
    if ((int)blockIdx.x < P.n_rg * P.n_kt) {
      const int rg = blockIdx.x / P.n_kt, kt = blockIdx.x % P.n_kt;
      const int nbc = min(kRouterTileChunks, P.n_rc - kRouterTileChunks * kt);
      prefetch_l2(P.router + ((int64_t)rg * P.n_ks * 64 + kRouterTileChunks * 32 * kt) * kRows * 16,
                  (uint32_t)(nbc * chunk_bytes(MOE_F32, kRouterCc)));
    }
    pend[0] = 0;
    for (int i = 0; i < P.n_stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], kConsumerWarps);
    }
    for (int i = 0; i < kRedSlots; ++i) {
      mbar_init(&rfull[i], kConsumerWarps);
      mbar_init(&rempty[i], 1);
    }
    mbar_init(reinterpret_cast<uint64_t*>(smem + plan.ebar), 1);
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  griddep_wait();  // x, the workspace and its counters are the previous launches' to finish with
  if (threadIdx.x == 0) {
    stamp_first_at(P.stamps, kTsEntry, t_entry);
    stamp_first(P.stamps, kTsStart);
  }
  __syncthreads();

  const int warp = threadIdx.x >> 5;
  if (warp == kProducerWarp) {
    if ((threadIdx.x & 31) == 0) producer_loop<L>(P, smem, plan);
  } else if (warp == kEpilogueWarp) {
    epilogue_loop<L>(P, smem, plan);
  } else {
    consumer_loop<L>(P, smem, plan);
  }

  __syncthreads();
  if (pend[0] > 0) {
    combine_blocks<L>(P, smem, plan, pend);
    __syncthreads();
    if (threadIdx.x == 0) stamp_last(P.stamps, kTsLastCombine);
  }
  // the last CTA out resets the cross-CTA counters for the next launch
  __syncthreads();
  if (threadIdx.x == 0) {
    stamp_first(P.stamps, kTsFirstExit);
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
    for (int i = threadIdx.x; i < P.n_dt; i += blockDim.x) P.d_cnt[i] = 0;
    for (int i = threadIdx.x; i < P.E_pad * P.Tp; i += blockDim.x) P.lfx[i] = 0;
    // this launch's phase stamps become the last completed launch's
    if (threadIdx.x < kNumStamps) {
      const unsigned long long v =
          threadIdx.x == kTsLastExit ? (unsigned long long)globaltimer_ns() : __ldcg(P.stamps + threadIdx.x);
      P.stamps[kNumStamps + threadIdx.x] = v;
      P.stamps[threadIdx.x] = 0ull;
    }
    if (threadIdx.x == 0) {
      P.sync->queue = 0;
      P.sync->router_done = 0;
      P.sync->x_done = 0;
      P.sync->routing_ready = 0;
      P.sync->routing_aux = 0;
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
  return smem_plan(P.n_stages, P.ring_bytes, P.misc_bytes, P.w_max).total;
}

cudaError_t small_t_configure(int L, int smem_bytes) {
  if (L == 2)
    return cudaFuncSetAttribute(moe_small_t_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
  return cudaFuncSetAttribute(moe_small_t_kernel<4>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem_bytes);
}

// Launched with programmatic stream serialization: the kernel may start while
// the previous kernel in the stream finishes (it waits for it before reading
// anything that kernel could have written).
cudaError_t small_t_launch(const SmallParams& P, int L, int grid, int smem_bytes, cudaStream_t st) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = (size_t)smem_bytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (L == 2) return cudaLaunchKernelEx(&cfg, moe_small_t_kernel<2>, P);
  return cudaLaunchKernelEx(&cfg, moe_small_t_kernel<4>, P);
}

}  // namespace moe
