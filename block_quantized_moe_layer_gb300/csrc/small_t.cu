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
// Work items, in order (each kind only waits on kinds before it, so every
// item another item waits for has already been taken by a running CTA):
//   router tiles     32 experts x 512 columns; each adds its share of the
//                    logits to a global sum kept as exact 2^-32 fixed point,
//                    with a count of the shares in the word's low bits
//                    (integer atomics, so the sum does not depend on the
//                    order of arrival, and a word says when it is complete).
//                    The tiles of the first 32 experts also write the
//                    activation records of their slice of x.  The routing
//                    (top-k, gates, permutation, expert work entries) is
//                    computed by the last CTA, which has no router tile,
//                    as soon as it reads complete words (or, with as many
//                    router tiles as CTAs, by the last router tile's CTA).
//   shared gate/up   32 outputs (16+16 gate/up rows, twice) x full K
//   routed gate/up   per routed work entry (<= 4 tokens of one expert)
//   shared down      128 outputs x full I
//   routed down
// Block b takes item b; every later item is claimed from one global queue.  A down tile's producer waits
// for its inputs (the entry's gate/up outputs) before it copies them, so the
// shared down tiles come after the routed gate/up ones: claimed earlier they
// would hold their producers (and leave their rings empty) until the shared
// gate/up finishes.  Before it waits for the previous kernel in the stream,
// block b copies the weights of its first stage (router tile b or a shared
// gate/up tile: constant data) and runs the router tile's code once, so that
// the code is warm when the slice of x arrives.
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
#include "gemv.cuh"
#include "layer.cuh"

namespace moe {

enum TileKind : int { kRouter = 0, kGateUp = 1, kDown = 2, kEnd = 3 };

struct Desc {
  int kind, chunk, nch, M;         // read by every consumer thread
  int nbc, fmt, rgks, off;         //   " (off = ring offset; rgks: router tiles: row
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
                      kSiteDrain = 7, kSiteRedEmpty = 8, kSiteRedFull = 9, kSiteLogits = 10 };

// Bounded spin on a global flag (acquire).  Returns false on timeout; the
// value seen goes to *seen when given.
__device__ inline bool wait_flag_geq(const int* p, int v, uint64_t limit_ns, int* status, int site, int detail,
                                     int* seen = nullptr) {
  int x = ld_acquire(p);
  if (x >= v) {
    if (seen) *seen = x;
    return true;
  }
  const uint64_t t0 = globaltimer_ns();
  int ns = 32;
  while (true) {
    x = ld_acquire(p);
    if (x >= v) {
      if (seen) *seen = x;
      return true;
    }
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

// Where a work item's stages come from and how large they are.  Shared by
// the prefetch before the dependency wait and the main loop, so both place
// and size the same stages.
struct Geo {
  int kind, rgk, rbt, entry, nbc, fmt, M, nch, ngroups, gps, need, nstages, slot0, n_tiles, e_id;
  uint32_t wb, per;
  int64_t cbytes;
  const uint8_t* wbase;
};

// A router tile: 32 experts (row group rg) x one 512-column slice rbt; one
// stage holding the tile's weights and then the slice of x.
template <int L>
__device__ __forceinline__ Geo geo_router(const SmallParams& P, int rg, int rbt) {
  constexpr int XEL = L == 2 ? 2 : 4;
  Geo g;
  g.kind = kRouter;
  g.rgk = rg << 16;
  g.rbt = rbt;
  g.entry = 0;
  g.nbc = min(kRouterTileChunks, P.n_rc - kRouterTileChunks * rbt);  // 128-column chunks in the slice
  g.fmt = MOE_F32;
  g.M = P.T;
  g.nch = 1;
  g.ngroups = 1;
  g.gps = 1;
  g.nstages = 1;
  g.slot0 = 0;
  g.n_tiles = 0;
  g.e_id = -1;
  g.cbytes = (int64_t)g.nbc * chunk_bytes(MOE_F32, kRouterCc);
  g.wbase = P.router + ((int64_t)rg * P.n_ks * 64 + kRouterTileChunks * 32 * rbt) * kRows * 16;
  g.wb = (uint32_t)g.cbytes;
  g.per = (uint32_t)(g.nbc * kRouterCc * XEL);
  g.need = (int)((g.wb + (uint32_t)g.M * g.per + 127u) & ~127u);
  return g;
}

// A gate/up tile (32 SwiGLU outputs: 16 gate + 16 up rows, twice) or a down
// tile (one 128-row block of z) of one work entry: the shared expert's
// (entry < n_sh) or a routed expert's (ep = its entry).
template <int L>
__device__ __forceinline__ Geo geo_expert(const SmallParams& P, int kind, int entry, int rbt, const Entry* ep) {
  constexpr int RB = rec_bytes(L);
  Geo g;
  g.kind = kind;
  g.rgk = 0;
  g.rbt = rbt;
  g.entry = entry;
  const bool shared_e = entry < P.n_sh;
  if (shared_e) {
    g.slot0 = P.T * P.k + kGroup * entry;
    g.M = min(kGroup, P.T - kGroup * entry);
    g.e_id = -1;
  } else {
    g.e_id = ep->e;
    g.slot0 = ep->slot0;
    g.M = ep->M;
  }
  g.fmt = shared_e ? P.sfmt : P.fmt;
  int kc;
  if (kind == kGateUp) {
    g.ngroups = 2;
    g.nch = shared_e ? P.sgu_nch : P.gu_nch;
    kc = shared_e ? P.sgu_kc : P.gu_kc;
    g.n_tiles = shared_e ? P.n_gu_sh : P.n_gu;
  } else {
    g.ngroups = 4;  // 128 output rows
    g.nch = shared_e ? P.sdn_nch : P.dn_nch;
    kc = shared_e ? P.sdn_kc : P.dn_kc;
    g.n_tiles = 0;
  }
  g.nbc = kc / 32;
  g.cbytes = chunk_bytes(g.fmt, kc);
  g.wbase = kind == kGateUp
                ? (shared_e ? P.sgu : P.gu + (int64_t)g.e_id * P.gu_stride) + (int64_t)(2 * rbt) * g.nch * g.cbytes
                : (shared_e ? P.sdn : P.dn + (int64_t)g.e_id * P.dn_stride) + (int64_t)(4 * rbt) * g.nch * g.cbytes;
  g.per = (uint32_t)(g.nbc * RB);
  // A group that is one chunk may share its stage with the next groups of
  // the tile (contiguous in memory, same records): fewer, larger stages,
  // as long as two of them fit the ring.
  g.gps = 1;
  if (g.nch == 1)
    while (2 * g.gps <= 4 && g.ngroups % (2 * g.gps) == 0 &&
           (int64_t)2 * g.gps * g.cbytes + (int64_t)g.M * g.per <= (int64_t)(P.ring_bytes / 2))
      g.gps *= 2;
  g.wb = (uint32_t)(g.gps * g.cbytes);
  g.need = (int)((g.wb + (uint32_t)g.M * g.per + 127u) & ~127u);
  g.nstages = g.ngroups * g.nch / g.gps;
  return g;
}

// Descriptor of stage q of an item, placed at ring offset pos.
__device__ __forceinline__ void write_desc(Desc* d, const Geo& g, int q, int pos) {
  const int grp = q * g.gps / g.nch, c = q * g.gps - grp * g.nch;
  const int kch = g.kind == kRouter ? kRouterTileChunks * g.rbt + c : 0;
  int4* dd = reinterpret_cast<int4*>(d);
  dd[0] = make_int4(g.kind, c, g.nch, g.M);
  dd[1] = make_int4(g.nbc, g.fmt, g.kind == kRouter ? g.rgk | kch : g.gps, pos);
  dd[2] = make_int4(g.entry, g.rbt, grp, g.ngroups);
  dd[3] = make_int4(g.slot0, 0, g.n_tiles, 0);
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
  const int NR = P.n_rg * P.n_kt;
  const int NDT = P.n_dt;  // down tiles per entry (128 output rows each)
  const int NSG = P.n_sh * P.n_gu_sh, NSD = P.n_sh * NDT;
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
  // Block b's first item is item b; later items are claimed from the
  // counter (offset by the grid), one ahead, so the claim's latency overlaps
  // the current item.  Claims on the one counter are served one at a time,
  // so the launch's first items, needed by every block at once, skip it.
  int t = blockIdx.x;
  while (ok) {
    const int t_next = (int)gridDim.x + atomicAdd(&P.sync->queue, 1);
    int kind = kGateUp, entry = 0, rbt = 0;
    if (t < NR) {
      kind = kRouter;
    } else if (t < NR + NSG) {
      entry = (t - NR) / P.n_gu_sh;
      rbt = (t - NR) % P.n_gu_sh;
    } else {
      if (n_rent < 0) {
        // the routing flag is published as 1 + the routed entry count
        int ready = 0;
        if (!wait_flag_geq(&P.sync->routing_ready, P.ready_target, P.timeout_ns, P.status, kSiteRouting, t, &ready)) {
          ok = false;
          break;
        }
        fence_proxy_async_global();
        n_rent = ready - 1;
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
      // routed gate/up, then the shared expert's down tiles (claimed once
      // every routed gate/up tile is, by when the shared gate/up outputs are
      // long written: a down tile claimed before its inputs exist would hold
      // its producer until they do), then routed down
      const int A = NR + NSG;
      const int NG = n_rent * P.n_gu, ND = n_rent * NDT;
      if (t < A + NG) {
        entry = P.n_sh + (t - A) / P.n_gu;
        rbt = (t - A) % P.n_gu;
      } else if (t < A + NG + NSD) {
        kind = kDown;
        entry = (t - A - NG) / NDT;
        rbt = (t - A - NG) % NDT;
      } else if (t < A + NG + NSD + ND) {
        kind = kDown;
        entry = P.n_sh + (t - A - NG - NSD) / NDT;
        rbt = (t - A - NG - NSD) % NDT;
      } else {
        stamp_last(P.stamps, kTsLastIssue);
        break;  // queue exhausted
      }
    }
    const Geo g = kind == kRouter ? geo_router<L>(P, t / P.n_kt, t % P.n_kt)
                                  : geo_expert<L>(P, kind, entry, rbt, ecache + entry);
    const bool xslice = g.kind == kRouter;  // the stage holds a slice of x
    const bool shared_e = g.kind != kRouter && g.entry < P.n_sh;
    // activation sources of this tile at chunk 0, and their step per chunk
    const uint8_t* asrc[kMaxSmallT];
    int64_t astep;
    if (xslice) {
      astep = 0;
#pragma unroll
      for (int m = 0; m < kMaxSmallT; ++m)
        asrc[m] = static_cast<const uint8_t*>(P.x) +
                  ((int64_t)m * P.H + (int64_t)kRouterTileChunks * g.rbt * kRouterCc) * XEL;
    } else {
      astep = (int64_t)g.nbc * RB;
      const Entry* ep = ecache + g.entry;
#pragma unroll
      for (int m = 0; m < kMaxSmallT; ++m) {
        const int mm = m < kGroup ? m : 0;
        asrc[m] = g.kind == kGateUp
                      ? P.xrec + (int64_t)(shared_e ? kGroup * g.entry + mm : ep->tok[mm]) * (P.H / 32) * RB
                      : P.hrec + (int64_t)(g.slot0 + mm) * (P.Imax / 32) * RB;
      }
    }
    bool dep_ok = xslice;
    if (g.kind == kGateUp && shared_e) {
      // the shared expert's records are read once they exist: the first row
      // group's router tiles write them before they count themselves done
      dep_ok = wait_flag_geq(&P.sync->router_done, P.n_rg * P.n_kt, P.timeout_ns, P.status, kSiteX, t);
      if (dep_ok) fence_proxy_async_global();
      else ok = false;
    }
    if (g.e_id >= 0) {
      if (g.kind == kGateUp && !st_gu) {
        stamp_first(P.stamps, kTsFirstRoutedIssue);
        st_gu = true;
      } else if (g.kind == kDown && !st_dn) {
        stamp_first(P.stamps, kTsFirstDownIssue);
        st_dn = true;
      }
    }
    for (int q = 0; q < g.nstages && ok; ++q) {
      const int grp = q * g.gps / g.nch, c = q * g.gps - grp * g.nch;
      // ring space: a free slot, then free bytes
      while (ok && issued - oldest >= NS) ok = wait_released(empty, NS, oldest++, P);
      int pos = 0;
      while (ok) {
        pos = head + g.need <= P.ring_bytes ? head : 0;
        if (oldest == issued) break;
        const int A = descs[oldest & (NS - 1)].off;
        if (A < head ? (pos + g.need <= A || pos >= head) : (pos >= head && pos + g.need <= A)) break;
        ok = wait_released(empty, NS, oldest++, P);
      }
      if (!ok) break;
      head = pos + g.need;
      const int s = issued & (NS - 1);
      uint8_t* stage = smem + plan.ring + pos;
      // (a block's first stage: its descriptor and weights were issued before
      // the dependency wait)
      if (!(issued == 0 && (int)blockIdx.x < NR + NSG)) {
        write_desc(descs + s, g, q, pos);
        mbar_arrive_expect_tx(&full[s], g.wb + (uint32_t)g.M * g.per);
        if (g.wb) bulk_g2s_hint(stage, g.wbase + (int64_t)q * g.wb, g.wb, &full[s], wpol);
      }
      if (!dep_ok) {
        if (g.kind == kGateUp) {
          dep_ok = true;  // routed gate/up: gated by the routing flag (shared: waited above)
        } else if (readybits[g.entry >> 5] & (1u << (g.entry & 31))) {
          dep_ok = true;
        } else {
          dep_ok = wait_flag_geq(&P.entry_ready[g.entry], 1, P.timeout_ns, P.status, kSiteEntry,
                                 g.entry * 65536 + (t & 0xFFFF));
          if (dep_ok) readybits[g.entry >> 5] |= 1u << (g.entry & 31);
        }
        if (dep_ok) fence_proxy_async_global();
        else ok = false;  // the consumers see the status word; the stage is still completed below
      }
      uint8_t* adst = stage + g.wb;
      const int64_t aoff = (int64_t)c * astep;
#pragma unroll
      for (int m = 0; m < kMaxSmallT; ++m)
        if (m < g.M) bulk_g2s(adst + m * g.per, dep_ok ? asrc[m] + aoff : asrc[0], g.per, &full[s]);
      (void)grp;
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

// Batcher's odd-even merge sort network for N (a power of two) inputs, as a
// comparator list in its iterative schedule (Knuth, TAOCP vol. 3, 5.3.4):
// 63 comparators for N = 16, 191 for N = 32.
struct SortNet {
  int n;
  unsigned char a[192], b[192];
};
template <int N>
__host__ __device__ constexpr SortNet batcher_net() {
  SortNet s{};
  for (int p = 1; p < N; p <<= 1)
    for (int k = p; k >= 1; k >>= 1)
      for (int j = k % p; j + k < N; j += 2 * k)
        for (int i = 0; i < k && i + j + k < N; ++i)
          if ((i + j) / (2 * p) == (i + j + k) / (2 * p)) {
            s.a[s.n] = (unsigned char)(i + j);
            s.b[s.n] = (unsigned char)(i + j + k);
            ++s.n;
          }
  return s;
}

// Sorts N 64-bit values into descending order in registers: comparator I
// and then the rest, by recursion, so that every index is a compile-time
// constant (entries known to be 0 fold away).
template <int N, int I = 0>
__device__ __forceinline__ void sort_desc(uint64_t (&c)[N]) {
  constexpr SortNet net = batcher_net<N>();
  if constexpr (I < net.n) {
    constexpr int a = net.a[I], b = net.b[I];
    const uint64_t x = c[a], y = c[b];
    c[a] = x > y ? x : y;
    c[b] = x > y ? y : x;
    sort_desc<N, I + 1>(c);
  }
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

__host__ __device__ constexpr int pow2_at_least(int n) { return n <= 1 ? 1 : 2 * pow2_at_least((n + 1) / 2); }

// The k largest of one token's E logits by (value desc, index asc), one
// warp, with the gates (softmax over the k selected logits, the sum by a
// fixed shuffle tree), written in slot order.
//
// Logit word (e, t) holds 256 S + n: S is the fixed-point sum (bias plus
// router slices, in units of 2^-32) and n the number of slices added so far,
// each slice one integer atomic.  The warp reads the token's words until
// every one holds all n_kt slices (a bounded wait: false on timeout), so no
// other flag has to order the slices before the read.  Logit e is S rounded
// once to fp32.
//
// Lane l holds experts l, l + 32, ... (NPER of them) as 64-bit composites
// (order-preserving key of the value, then the complemented index, so a
// larger composite is a larger value or, on equal values, a lower index;
// 0 = none) and sorts them.  Each round takes the exact maximum of the
// lanes' heads (a warp max of the keys; if several lanes hold it, the lowest
// expert index among them wins by a second warp min, only then); the winning
// lane writes the slot and drops its head.
//
// This code runs once per launch, so its instructions are cold: the first
// read of the words, complete or not, also runs the selection (results
// overwritten later), so that the pass on the complete words finds it warm.
//
template <int NPER>
__device__ __forceinline__ bool topk_token(const SmallParams& P, int t, int* ids, float* vals, float* gates) {
  const int lane = threadIdx.x & 31;
  const int E = P.E, k = P.k;
  constexpr int NP = pow2_at_least(NPER);
  constexpr int NL = NP < kMaxTopK ? NP : kMaxTopK;  // (sorted lists) a lane wins at most k <= kMaxTopK rounds
  uint64_t t0 = 0;
  bool warm = false;
  while (true) {
    uint64_t c[NP];
    bool done = true;
#pragma unroll
    for (int i = 0; i < NP; ++i) {
      const int e = lane + 32 * i;
      c[i] = 0ull;
      if (i < NPER && e < E) {
        const long long w = ld_relaxed_s64(P.lfx + (int64_t)e * kMaxSmallT + t);
        if ((int)(w & 255) != P.n_kt) done = false;
        const float x = __ll2float_rn(w >> 8) * 0x1p-32f;
        c[i] = ((uint64_t)order_key(x) << 32) | (uint64_t)(~(uint32_t)e);
      }
    }
    done = __all_sync(0xffffffffu, done);
    if (done && t == 0 && lane == 0) stamp_last(P.stamps, kTsRouterDone);
    if (done || !warm) {
      // up to 16 per lane: sorted, the head dropped per win; more (E > 512):
      // unsorted, the lane's best found again by a tree per win (a 32-input
      // network needs more registers than the kernel has)
      uint64_t best = 0ull;
      if constexpr (NP <= 16) sort_desc(c);
      else best = tree_max(c);
#pragma unroll 1
      for (int j = 0; j < k; ++j) {
        const uint64_t b = NP <= 16 ? c[0] : best;
        const uint32_t key = (uint32_t)(b >> 32);
        const uint32_t m = __reduce_max_sync(0xffffffffu, key);
        const uint32_t holders = __ballot_sync(0xffffffffu, b != 0ull && key == m);
        int wl = __ffs(holders) - 1;
        if (holders & (holders - 1u))
          wl = (int)(__reduce_min_sync(0xffffffffu, (holders >> lane) & 1u ? ~(uint32_t)b : 0x7fffffffu) & 31u);
        const bool win = lane == wl;
        if (win) {
          ids[j] = (int)~(uint32_t)b;
          vals[j] = key_value(m);
        }
        if constexpr (NP <= 16) {
#pragma unroll
          for (int i = 0; i + 1 < NL; ++i) c[i] = win ? c[i + 1] : c[i];
          c[NL - 1] = win ? 0ull : c[NL - 1];
        } else if (win) {
          const int slot = (int)((~(uint32_t)b) >> 5);
#pragma unroll
          for (int i = 0; i < NP; ++i)
            if (i == slot) c[i] = 0ull;
          best = tree_max(c);
        }
      }
      __syncwarp();
      const float l0 = vals[0];
      const float ex = lane < k ? expf(vals[lane] - l0) : 0.f;
      float sum = ex;
#pragma unroll
      for (int o = 16; o; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
      if (lane < k) gates[lane] = ex / sum;
      __syncwarp();
      if (done) break;
      warm = true;
    }
    int stop = 0;
    if (lane == 0) {
      const uint64_t now = globaltimer_ns();
      if (t0 == 0) t0 = now;
      if (now - t0 > P.timeout_ns) {
        record_timeout(P.status, kSiteLogits, t);
        stop = 1;
      } else if (ld_acquire(P.status) != 0) {
        stop = 1;
      }
    }
    if (__shfl_sync(0xffffffffu, stop, 0)) return false;
  }
  return true;
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

// Runs on the consumer threads of one CTA: logits, top-k and gates, then the
// permutation and the routed work entries.  Polled (the usual case: fewer
// router tiles than CTAs): the last CTA, which has no router tile, runs it
// as soon as every logit word holds all its slices; it acquires the router
// count only to publish the x records with the routing.  Otherwise the CTA
// that counted the last router tile runs it (the count orders the slices).  The entries and their count are published first (routing_ready);
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
__device__ __forceinline__ void finalize_routing(const SmallParams& P, uint8_t* misc, int* pend, bool polled) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  constexpr int NT = kConsumerWarps * 32;
  const int T = P.T, E = P.E, k = P.k, Tk = P.T * P.k;
  const FinLayout f = fin_layout(T, E, k);
  int* sid = reinterpret_cast<int*>(misc + f.sid);      // [Tk]
  float* sl = reinterpret_cast<float*>(misc + f.sl);    // [Tk]
  float* sg = reinterpret_cast<float*>(misc + f.sg);    // [Tk]
  int* sperm = reinterpret_cast<int*>(misc + f.sperm);  // [Tk]
  int* spos = reinterpret_cast<int*>(misc + f.spos);    // [Tk]
  int* slt = reinterpret_cast<int*>(misc + f.slt);      // [Tk] pairs of lower experts
  int* srank = reinterpret_cast<int*>(misc + f.srank);  // [Tk] earlier pairs of the same expert
  int* sent = reinterpret_cast<int*>(misc + f.sent);    // [Tk] entries owned (first pair of an expert)

  // top-k and gates per token, one warp per token, straight from the
  // fixed-point logit sums
  bool ok = true;
  #pragma unroll 1
  for (int t = warp; t < T; t += kConsumerWarps) {
    bool r;
    if (E <= 128) r = topk_token<4>(P, t, sid + t * k, sl + t * k, sg + t * k);
    else if (E <= 384) r = topk_token<12>(P, t, sid + t * k, sl + t * k, sg + t * k);
    else r = topk_token<kMaxE / 32>(P, t, sid + t * k, sl + t * k, sg + t * k);
    ok = ok && r;
  }
  // polled: a warp without a token (warp 0 after its own, at T = 8) acquires
  // the router count, so that thread 0's release of the routing below also
  // publishes the x records
  const int xw = T < kConsumerWarps ? T : 0;
  if (polled && warp == xw && lane == 0) {
    if (wait_flag_geq(&P.sync->router_done, P.n_rg * P.n_kt, P.timeout_ns, P.status, kSiteX, -1))
      stamp_last(P.stamps, kTsXDone);
    else
      ok = false;
  }
  if (consumer_sync_or(!ok)) return;  // a wait timed out: the status word says which
  // (stamps here come from warp 1: the release below is thread 0's, and a
  // release waits for its own thread's earlier writes)
  if (tid == 32) stamp_last(P.stamps, kTsTopkDone);

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
  if (tid == 32) stamp_last(P.stamps, kTsEntriesDone);
  if (tid == 0) {
    P.sync->n_rent = n_rent;
    st_release(&P.sync->routing_ready, 1 + n_rent);
    stamp_last(P.stamps, kTsRoutingReady);
    *nrent_s = n_rent;
  }
  consumer_sync();
  // One arrival of the routing on every 128-row block of z: a block is
  // complete after the down tile of each of the n_sh + n_rent entries and
  // this arrival, and whoever arrives last combines it.  A shared down tile that finishes before the
  // routing is known can therefore never be taken for the last one, and a
  // layer with no down work for this batch (a shard none of whose experts
  // was chosen, with no shared expert) still gets y from the combine.
  {
    const int last = P.n_sh + *nrent_s;
    for (int b = tid; b < P.n_dt; b += NT)
      if (atom_add_acq_rel(&P.d_cnt[b], 1) == last) pend[1 + atomicAdd(&pend[0], 1)] = b;
  }
  // The logit sums were read by this block only (the top-k, above): restore
  // them to their starting value (the bias) for the next launch now, off the
  // launch's tail.  Thread i takes experts i, i + 256, ...: one read of the
  // bias table, then the expert's 8 token columns.
  for (int e = tid; e < P.E_pad; e += NT) {
    const long long v = P.lfx0[e];
    longlong2* row = reinterpret_cast<longlong2*>(P.lfx + (int64_t)e * kMaxSmallT);
#pragma unroll
    for (int q = 0; q < kMaxSmallT / 2; ++q) row[q] = make_longlong2(v, v);
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
// accumulators per token (one per float4 component).  A full 512-column
// slice loads its columns in batches (weights and x first, then the FMAs),
// so that the shared-memory latency is paid once per batch.
template <int L, int T>
__device__ __forceinline__ void router_dot(const float4* wst, const uint8_t* xs, int cols, float (&racc)[kMaxSmallT]) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  constexpr int XEL = L == 2 ? 2 : 4;
  float ra[T][4];
#pragma unroll
  for (int t = 0; t < T; ++t)
#pragma unroll
    for (int c = 0; c < 4; ++c) ra[t][c] = 0.f;
  auto fma4 = [&](const float4& w, const uint8_t* xp, int t) {
    float4 xv;
    if constexpr (L == 2) {
      const uint2 raw = *reinterpret_cast<const uint2*>(xp);
      xv = make_float4(__uint_as_float(raw.x << 16), __uint_as_float(raw.x & 0xFFFF0000u), __uint_as_float(raw.y << 16),
                       __uint_as_float(raw.y & 0xFFFF0000u));
    } else {
      xv = *reinterpret_cast<const float4*>(xp);
    }
    ra[t][0] = fmaf(w.x, xv.x, ra[t][0]);
    ra[t][1] = fmaf(w.y, xv.y, ra[t][1]);
    ra[t][2] = fmaf(w.z, xv.z, ra[t][2]);
    ra[t][3] = fmaf(w.w, xv.w, ra[t][3]);
  };
  if (cols == kRouterTileChunks * kRouterCc) {
    constexpr int NI = kRouterTileChunks * kRouterCc / 4 / kConsumerWarps;  // 16 columns of float4 per warp
    constexpr int B = (T <= 4 && L == 2) ? 8 : 4;                            // columns per batch
#pragma unroll
    for (int h = 0; h < NI / B; ++h) {
      float4 w[B];
      uint4 xr[B][T];  // the x values of column group k4 (8 or 16 bytes per token)
#pragma unroll
      for (int i = 0; i < B; ++i) {
        const int k4 = warp + kConsumerWarps * (B * h + i);
        w[i] = wst[k4 * 32 + lane];
#pragma unroll
        for (int t = 0; t < T; ++t) {
          if constexpr (L == 2) {
            const uint2 r = *reinterpret_cast<const uint2*>(xs + (t * cols + k4 * 4) * XEL);
            xr[i][t] = make_uint4(r.x, r.y, 0u, 0u);
          } else {
            xr[i][t] = *reinterpret_cast<const uint4*>(xs + (t * cols + k4 * 4) * XEL);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < B; ++i)
#pragma unroll
        for (int t = 0; t < T; ++t) fma4(w[i], reinterpret_cast<const uint8_t*>(&xr[i][t]), t);
    }
  } else {
    const int ncol4 = cols / 4;
#pragma unroll 4
    for (int i = 0; i < 16; ++i) {
      const int k4 = warp + kConsumerWarps * i;
      if (k4 < ncol4) {
        const float4 w = wst[k4 * 32 + lane];
#pragma unroll
        for (int t = 0; t < T; ++t) fma4(w, xs + (t * cols + k4 * 4) * XEL, t);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kMaxSmallT; ++t) racc[t] = t < T ? (ra[t][0] + ra[t][1]) + (ra[t][2] + ra[t][3]) : 0.f;
}

struct RouterAcc {
  float v[kMaxSmallT];
};

// One router tile's dot products for T tokens (runtime).  Not inlined: a
// router CTA runs this code once per launch, so its instructions are cold;
// its consumer warps call it once on the stage before the dependency wait
// (weights in flight, x not there yet, results discarded) and then find it
// warm for the real call.
template <int L>
__device__ __noinline__ RouterAcc router_tile_dot(const float4* wst, const uint8_t* xs, int cols, int T) {
  RouterAcc r;
  switch (T) {
    case 1: router_dot<L, 1>(wst, xs, cols, r.v); break;
    case 2: router_dot<L, 2>(wst, xs, cols, r.v); break;
    case 3: router_dot<L, 3>(wst, xs, cols, r.v); break;
    case 4: router_dot<L, 4>(wst, xs, cols, r.v); break;
    case 5: router_dot<L, 5>(wst, xs, cols, r.v); break;
    case 6: router_dot<L, 6>(wst, xs, cols, r.v); break;
    case 7: router_dot<L, 7>(wst, xs, cols, r.v); break;
    default: router_dot<L, 8>(wst, xs, cols, r.v); break;
  }
  return r;
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
  // With fewer router tiles than CTAs the last CTA has none (its items are
  // all claimed past the router's); it routes first, polling the logits.
  const bool polled = P.n_rg * P.n_kt < (int)gridDim.x;
  if (polled && blockIdx.x == gridDim.x - 1) finalize_routing(P, misc, reinterpret_cast<int*>(smem + plan.pend), true);

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

    if (d.kind == kRouter) {
      // One router tile: 32 experts (lane = expert row) x a slice of ncc
      // 128-column chunks.  The stage holds the tile's router weights
      // ([cols/4][32 rows][4]) and then the slice of x ([T][cols]).
      const int ncc = d.nbc, cols = ncc * kRouterCc;
      const float4* wst = reinterpret_cast<const float4*>(stage);
      const uint8_t* xs = stage + cols * kRows * 4;
      {
        const RouterAcc r = router_tile_dot<L>(wst, xs, cols, T);
#pragma unroll
        for (int t = 0; t < kMaxSmallT; ++t) racc[t] = r.v[t];
      }
#pragma unroll
      for (int t = 0; t < kMaxSmallT; ++t)
        if (t < T) rred[(warp * kMaxSmallT + t) * 32 + lane] = racc[t];
      consumer_sync();
      if (tid < T * 32) {
        // this slice's share of logit (t, expert 32 rg + r), added as an
        // exact integer multiple of 2^-32 to a sum that starts from the bias,
        // together with one count in the word's low 8 bits: the total does
        // not depend on the order in which the slices arrive, and the word
        // says by itself when it is complete.  A share saturates at 2^17 in
        // magnitude (a NaN share counts as -2^17), so that n_kt <= 32 slices
        // and the bias never overflow the word.
        const int t = tid >> 5, r = tid & 31;
        float v = 0.f;
        for (int w = 0; w < kConsumerWarps; ++w) v += rred[(w * kMaxSmallT + t) * 32 + r];
        const float q = fminf(fmaxf(v * 4294967296.f, -0x1p49f), 0x1p49f);
        atomicAdd(reinterpret_cast<unsigned long long*>(P.lfx) + (int64_t)(d_rg * 32 + r) * kMaxSmallT + t,
                  ((unsigned long long)__float2ll_rn(q) << 8) + 1ull);
      }
      if (d_rg == 0) {
        // after the logit shares (they start the routing): the first row
        // group's tiles also turn their slice of x into the activation
        // records, one 32-column block per thread from warp 4 on; the proxy
        // fence makes them visible to the bulk copies that read them once
        // every router tile has counted itself done
        const int kt = d_ks / kRouterTileChunks, nb = cols / 32;
        constexpr int XEL = L == 2 ? 2 : 4;
        const int i = tid - 4 * 32;
        if (i >= 0 && i < T * nb) {
          const int t = i / nb, b = i - (i / nb) * nb;
          write_record_lane<L>(xs + (t * cols + b * 32) * XEL,
                               P.xrec + ((int64_t)t * (P.H / 32) + kt * (kRouterTileChunks * kRouterCc / 32) + b) * RB);
          fence_proxy_async_global();
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[s]);  // the stage (weights, x slice) is read
      // the barrier orders every thread's record writes (and additions)
      // before thread 0's release count, which the shared expert's records
      // and, through the routing, the routed tiles' records wait for
      consumer_sync();
      if (polled) {
        // the routing CTA reads the logit words by themselves; the count
        // publishes this tile's x records
        if (tid == 0) red_add_release(&P.sync->router_done, 1);
      } else {
        if (tid == 0) {
          const int old = atom_add_acq_rel(&P.sync->router_done, 1);
          flags[0] = (old == P.n_rg * P.n_kt - 1);
        }
        consumer_sync();
        if (flags[0]) {
          if (tid == 32) stamp_last(P.stamps, kTsXDone);  // the x records are written by router tiles
          finalize_routing(P, misc, reinterpret_cast<int*>(smem + plan.pend), false);
        }
        consumer_sync();
      }
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
        gemv_chunk<L>(stage + j * cb, recs, d.nbc, d.fmt, j, d.M, acc);
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

// The combine's routing arrays in shared memory, by one warp: gates and z
// positions of the T*k pairs (position -1 for a pair whose expert another
// shard holds).  Waits (bounded) for the routing arrays to be published;
// returns false on timeout.
__device__ bool preload_routing(const SmallParams& P, uint8_t* smem, const SmemPlan& plan) {
  float* sg = reinterpret_cast<float*>(smem + plan.escr);                          // [T*k] gates
  int* sp = reinterpret_cast<int*>(smem + plan.escr + kMaxSmallT * kMaxTopK * 4);  // [T*k] slots
  int ok = 0;
  if ((threadIdx.x & 31) == 0) ok = wait_flag_geq(&P.sync->routing_aux, 1, P.timeout_ns, P.status, kSiteRouting, -1);
  ok = __shfl_sync(0xffffffffu, ok, 0);
  if (!ok) return false;
  for (int q = threadIdx.x & 31; q < P.T * P.k; q += 32) {
    const int e = __ldcg(&P.ids[q]);
    sg[q] = __ldcg(&P.gates[q]);
    sp[q] = e >= P.e0 && e < P.e0 + P.n_e ? __ldcg(&P.pos[q]) : -1;
  }
  __syncwarp();
  return true;
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
  bool preloaded = false;
  int n_rent_c = -1;  // (lane 0) routed entries, once known
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
      if (!preloaded && d.entry >= P.n_sh) {
        // the first routed down tile: the routing is published (and its
        // arrays follow right after), so fetch what a combine of this block
        // needs now rather than when the block completes
        preloaded = true;
        if (preload_routing(P, smem, plan) && lane == 0) reinterpret_cast<int*>(smem + plan.flags)[3] = 1;
      }
      const int row = d.rbt * 128 + d.group * 32 + lane;
      for (int m = 0; m < d.M; ++m) P.z[(int64_t)(d.slot0 + m) * P.H + row] = v[m];
      if (d.group == d.ngroups - 1) {
        __syncwarp();  // orders the lanes' z writes before lane 0's release
        if (lane == 0) {
          // The block is complete after every entry's down tile (n_sh +
          // n_rent) and the routing's own arrival, which comes after the
          // routing is published.  So a tile whose increment finds the block
          // complete has acquired the routing; it reads n_rent after the
          // increment (once per block of this CTA: then it is cached).  Until
          // the routing has arrived no tile can be the last one.
          const int blk = d.rbt;
          const int old = atom_add_acq_rel(&P.d_cnt[blk], 1);
          if (n_rent_c < 0 && (d.entry >= P.n_sh || ld_acquire(&P.sync->routing_ready)))
            n_rent_c = ld_acquire(&P.sync->n_rent);
          if (n_rent_c >= 0 && old == P.n_sh + n_rent_c) {
            stamp_last(P.stamps, kTsLastDownDone);
            // this CTA combines the block when it leaves (with all its threads)
            int* pend = reinterpret_cast<int*>(smem + plan.pend);
            pend[1 + atomicAdd(&pend[0], 1)] = blk;
          }
        }
      }
    }
  }
}

// y rows of the 128-row blocks this CTA completed last, in slot order:
// y[t] = sum_{j<k} g[t,j] z[pos[t,j]] + z_shared[t], all threads of the CTA.
// The z rows of other blocks' tiles were released by their down-count
// increments and acquired by this CTA's own; the CTA barrier before this
// call passes that on to every thread.
template <int L>
__device__ void combine_blocks(const SmallParams& P, uint8_t* smem, const SmemPlan& plan, const int* pend) {
  const float* sg = reinterpret_cast<const float*>(smem + plan.escr);
  const int* sp = reinterpret_cast<const int*>(smem + plan.escr + kMaxSmallT * kMaxTopK * 4);
  const int T = P.T, k = P.k;
  int* flags = reinterpret_cast<int*>(smem + plan.flags);
  if (threadIdx.x == 0) stamp_last(P.stamps, kTsCombineStart);
  if (!flags[3]) {
    // not fetched by the epilogue warp (this CTA saw no routed down tile)
    if (threadIdx.x < 32) {
      const bool ok = preload_routing(P, smem, plan);
      if (threadIdx.x == 0) flags[2] = ok;
    }
    __syncthreads();
    if (!flags[2]) return;
  }
  if (threadIdx.x == 0) stamp_last(P.stamps, kTsCombineReady);
  // one pass: thread u takes 4 consecutive rows of one token of one block,
  // with all of its z reads (128-bit) in flight at once
  const int n = pend[0];
  for (int u = threadIdx.x; u < n * 32 * T; u += blockDim.x) {
    const int b = u / (32 * T), rem = u - b * (32 * T), t = rem / 32;
    const int r = pend[1 + b] * 128 + (rem - t * 32) * 4;
    float4 zv[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k && sp[t * k + j] >= 0) zv[j] = __ldcg(reinterpret_cast<const float4*>(P.z + (int64_t)sp[t * k + j] * P.H + r));
    const float4 zs = P.n_sh > 0 ? __ldcg(reinterpret_cast<const float4*>(P.z + (int64_t)(T * k + t) * P.H + r))
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (j < k && sp[t * k + j] >= 0) {
        const float g = sg[t * k + j];
        acc.x = fmaf(g, zv[j].x, acc.x);
        acc.y = fmaf(g, zv[j].y, acc.y);
        acc.z = fmaf(g, zv[j].z, acc.z);
        acc.w = fmaf(g, zv[j].w, acc.w);
      }
    acc.x += zs.x;
    acc.y += zs.y;
    acc.z += zs.z;
    acc.w += zs.w;
    const int64_t o = (int64_t)t * P.H + r;
    if (P.h_in) {
      // residual-stream mode: h_out = h_in + y in fp32 (h_in may be h_out),
      // and this block's sum of squares of token t's row.  A warp's 32 lanes
      // are one (block, token) here (32 units each; the CTA has whole
      // warps), summed by a fixed shuffle tree.
      const float4 hv = *reinterpret_cast<const float4*>(P.h_in + o);
      acc.x += hv.x;
      acc.y += hv.y;
      acc.z += hv.z;
      acc.w += hv.w;
      *reinterpret_cast<float4*>(P.h_out + o) = acc;
      float q = fmaf(acc.w, acc.w, fmaf(acc.z, acc.z, fmaf(acc.y, acc.y, acc.x * acc.x)));
#pragma unroll
      for (int off = 16; off; off >>= 1) q += __shfl_xor_sync(0xffffffffu, q, off);
      if ((threadIdx.x & 31) == 0) P.ssq[t * P.n_dt + pend[1 + b]] = q;
      continue;
    }
    if (P.residual) {
      if constexpr (L == 2) {
        const uint2 xr = *reinterpret_cast<const uint2*>(reinterpret_cast<const __nv_bfloat16*>(P.x) + o);
        acc.x += __uint_as_float(xr.x << 16);
        acc.y += __uint_as_float(xr.x & 0xFFFF0000u);
        acc.z += __uint_as_float(xr.y << 16);
        acc.w += __uint_as_float(xr.y & 0xFFFF0000u);
      } else {
        const float4 xr = *reinterpret_cast<const float4*>(reinterpret_cast<const float*>(P.x) + o);
        acc.x += xr.x;
        acc.y += xr.y;
        acc.z += xr.z;
        acc.w += xr.w;
      }
    }
    if (L == 2 && !P.out_f32) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(P.y) + o) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    } else {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(P.y) + o) = acc;
    }
  }
}

// Residual-stream mode, after this CTA combined `nb` blocks (all threads):
// the CTA whose blocks complete the set normalises the rows,
// xn[t] = h_out[t] / sqrt(mean(h_out[t]^2) + eps), from the blocks' sums of
// squares taken in block order.  The other CTAs' h_out and sums were
// released by their count increments (after a CTA barrier) and are acquired
// by this CTA's own.
template <int L>
__device__ void norm_rows(const SmallParams& P, uint8_t* smem, const SmemPlan& plan, int nb) {
  int* flags = reinterpret_cast<int*>(smem + plan.flags);
  float* inv = reinterpret_cast<float*>(smem + plan.rred);  // free at this point
  if (threadIdx.x == 0) {
    const int old = atom_add_acq_rel(&P.sync->norm_cnt, nb);
    flags[12] = (old + nb == P.n_dt);
  }
  __syncthreads();
  if (!flags[12]) return;
  if (threadIdx.x < P.T) {
    float sq = 0.f;
    for (int b = 0; b < P.n_dt; ++b) sq += __ldcg(P.ssq + threadIdx.x * P.n_dt + b);
    inv[threadIdx.x] = 1.f / sqrtf(sq / (float)P.H + P.eps);
  }
  __syncthreads();
  const int q4 = P.H / 4;
  for (int u = threadIdx.x; u < P.T * q4; u += blockDim.x) {
    const int t = u / q4;
    const int64_t o = (int64_t)t * P.H + (int64_t)(u - t * q4) * 4;
    const float4 h = __ldcg(reinterpret_cast<const float4*>(P.h_out + o));
    const float s = inv[t];
    if constexpr (L == 2) {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(h.x * s, h.y * s), hi = __floats2bfloat162_rn(h.z * s, h.w * s);
      *reinterpret_cast<uint2*>(reinterpret_cast<__nv_bfloat16*>(P.xn) + o) =
          make_uint2(*reinterpret_cast<const uint32_t*>(&lo), *reinterpret_cast<const uint32_t*>(&hi));
    } else {
      *reinterpret_cast<float4*>(reinterpret_cast<float*>(P.xn) + o) = make_float4(h.x * s, h.y * s, h.z * s, h.w * s);
    }
  }
  if (threadIdx.x == 0) P.sync->norm_cnt = 0;  // every CTA has counted: ready for the next launch
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
    pend[0] = 0;
    flags[3] = 0;  // the combine's routing arrays are not in shared memory yet
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
  __syncthreads();
  // constant data only: the weights of this block's first stage (its first
  // item, a router tile or a shared gate/up tile, stage 0 at ring offset 0)
  // are copied before the dependency wait, while the previous launch ends;
  // the producer adds the activations to the same stage after it
  const int n_early = P.n_rg * P.n_kt + P.n_sh * P.n_gu_sh;
  if (threadIdx.x == kProducerWarp * 32 && (int)blockIdx.x < n_early) {
    const int b = blockIdx.x, nr = P.n_rg * P.n_kt;
    const Geo g = b < nr ? geo_router<L>(P, b / P.n_kt, b % P.n_kt)
                         : geo_expert<L>(P, kGateUp, (b - nr) / P.n_gu_sh, (b - nr) % P.n_gu_sh, nullptr);
    // the descriptor first: the arrival below releases it to the consumers
    write_desc(reinterpret_cast<Desc*>(smem + plan.descs), g, 0, 0);
    mbar_arrive_expect_tx(&full[0], g.wb + (uint32_t)g.M * g.per);
    bulk_g2s_hint(smem + plan.ring, g.wbase, g.wb, &full[0], l2_evict_first_policy());
  } else if ((threadIdx.x >> 5) < kConsumerWarps && (int)blockIdx.x < P.n_rg * P.n_kt) {
    // warm the router tile's code on the stage (its bytes still arriving;
    // the result is discarded, only its instructions are wanted)
    const int cols = min(kRouterTileChunks, P.n_rc - kRouterTileChunks * ((int)blockIdx.x % P.n_kt)) * kRouterCc;
    const RouterAcc r = router_tile_dot<L>(reinterpret_cast<const float4*>(smem + plan.ring),
                                           smem + plan.ring + cols * kRows * 4, cols, P.T);
    asm volatile("" ::"f"(r.v[0]));
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
    if (P.h_in) norm_rows<L>(P, smem, plan, pend[0]);
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
      P.sync->routing_ready = 0;
      P.sync->routing_aux = 0;
      P.sync->n_rent = 0;
      P.sync->exit_cnt = 0;
    }
    // (no fence: the grid's completion makes these writes visible to the
    // next launch, whose dependency wait waits for it)
  }
}

// ---------------------------------------------------------------------------
// host side
// ---------------------------------------------------------------------------
// The router logit words' starting value: the bias in units of 2^-32 (exact
// for |b| >= 2^-8, rounded to the nearest 2^-32 below that; saturated at
// 2^17 in magnitude), times 256 (no slices counted yet), written to the
// table lfx0 and to every token column of lfx.
__global__ void logit_sums_init_kernel(const float* __restrict__ bias, int E, int E_pad, long long* __restrict__ lfx0,
                                       long long* __restrict__ lfx) {
  const int i = blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= E_pad * kMaxSmallT) return;
  const int e = i / kMaxSmallT;
  const float q = (bias && e < E) ? fminf(fmaxf(bias[e] * 4294967296.f, -0x1p49f), 0x1p49f) : 0.f;
  const long long v = (long long)((unsigned long long)__float2ll_rn(q) << 8);
  lfx[i] = v;
  if (i % kMaxSmallT == 0) lfx0[e] = v;
}

cudaError_t small_t_init_logit_sums(const SmallParams& P, long long* lfx0, cudaStream_t st) {
  const int n = P.E_pad * kMaxSmallT;
  logit_sums_init_kernel<<<(n + 255) / 256, 256, 0, st>>>(P.router_b, P.E, P.E_pad, lfx0, P.lfx);
  return cudaGetLastError();
}

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
