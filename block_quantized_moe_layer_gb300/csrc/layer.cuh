// layer.cuh -- the layer object and the parameter block of the small-T kernel.
#pragma once
#include "common.cuh"

namespace moe {

struct LtState;  // the prefill-sized path's weights and workspace (large_t.cu)

// One unit of expert work: up to kGroup activation vectors routed to one
// expert (e == -1 for the shared expert).  Slots index the activation /
// intermediate rows: routed slots are positions in perm[], the shared
// expert's slot for token t is T*k + t.
struct Entry {
  int e;
  int slot0;
  int M;
  int tok[kGroup];
  int pad;  // 32 bytes: copied with 16-byte loads
};
static_assert(sizeof(Entry) == 32, "Entry is copied as two 16-byte vectors");

// Cross-CTA counters of the fused kernel.  All zero between launches: the
// last CTA to leave resets them.  Each busy counter has an L2 line (128 B)
// of its own, so that the blocks polling one flag do not queue behind the
// atomics on another.
struct Sync {
  alignas(128) int queue;          // next tile to claim
  alignas(128) int router_done;    // router tiles finished (also: x records complete)
  alignas(128) int routing_ready;  // routing published: 1 + the routed entry count
  int n_rent;                      // routed entries (written with the routing)
  alignas(128) int routing_aux;    // ids, gates, offsets, perm, pos written (after routing_ready)
  alignas(128) int exit_cnt;       // CTAs that left
  alignas(128) int norm_cnt;       // residual-stream mode: 128-row blocks combined
};

// Phase stamps of one small-T launch (globaltimer, ns).  Each kind is kept
// in one 64-bit word of the workspace: "first" events as the maximum of the
// complemented time (so every word is an atomic maximum and starts at 0),
// "last" and single events as the maximum of the time.  The last CTA to
// leave copies the words to a second array (the last completed launch) and
// zeroes them; a launch's CTAs only write them after their dependency wait,
// so consecutive launches never mix.
enum Stamp : int {
  kTsEntry = 0,          // first: a CTA entered the kernel (before its dependency wait)
  kTsStart,              // first: a CTA passed the dependency wait
  kTsXDone,              // the x records are complete
  kTsRouterDone,         // the last router tile finished (the routing starts)
  kTsRoutingReady,       // the routing is published
  kTsFirstRoutedIssue,   // first: a routed gate/up weight copy is issued
  kTsFirstRoutedCompute, // first: a consumer starts a routed gate/up stage
  kTsSharedGateUp,       // last: the shared expert's gate/up outputs are complete
  kTsLastGateUp,         // last: a routed entry's gate/up outputs are complete
  kTsFirstDownIssue,     // first: a routed down weight copy is issued
  kTsLastIssue,          // last: a producer found the queue exhausted
  kTsLastDownDone,       // last: a 128-row block of z is complete
  kTsLastCombine,        // last: a combine finished
  kTsFirstExit,          // first: a CTA is leaving
  kTsLastExit,           // the last CTA is leaving
  kTsCombineStart,       // last: a combining CTA's roles are done (its combine starts)
  kTsCombineReady,       // last: a combining CTA has the routing arrays in shared memory
  kTsTopkDone,           // the routing's top-k and gates are done
  kTsEntriesDone,        // the routing's permutation and work entries are written
  kNumStamps
};
constexpr uint32_t kStampFirstMask = (1u << kTsEntry) | (1u << kTsStart) | (1u << kTsFirstRoutedIssue) |
                                     (1u << kTsFirstRoutedCompute) | (1u << kTsFirstDownIssue) |
                                     (1u << kTsFirstExit);

struct SmallParams {
  // shapes
  int H, E, k, I, Ish, T;
  int e0, n_e;            // routed experts held by this layer: [e0, e0 + n_e) (all E unless sharded)
  int n_rg, n_ks, n_kt;   // router: row groups of 32 experts, 256-column repack blocks, 512-column tiles
  int n_rc;               // router: 128-column chunks (H / 128)
  int Tp;                 // T rounded up to 4
  int n_gu, n_gu_sh;      // gate/up tiles per routed / shared entry (32 outputs each)
  int n_dt;               // down tiles per entry (128 outputs each; the unit of the combine)
  int n_sh;               // shared entries for this T
  int Imax;               // max(I, Ish): row stride of the h records
  int E_pad;              // n_rg * 32
  int w_max;              // capacity of the entry arrays
  // weights (repacked)
  const uint8_t* router;  // [n_rg][n_ks][32 rows x 256 cols fp32]
  const float* router_b;  // [E] or nullptr
  const uint8_t* gu;      // routed gate/up, expert stride gu_stride
  const uint8_t* dn;      // routed down, expert stride dn_stride
  const uint8_t* sgu;     // shared gate/up (nullptr if none)
  const uint8_t* sdn;     // shared down
  int64_t gu_stride, dn_stride;
  int fmt, sfmt;
  int gu_nch, gu_kc, dn_nch, dn_kc, sgu_nch, sgu_kc, sdn_nch, sdn_kc;
  // activations
  const void* x;  // [T, H] bf16 (L = 2) or fp32 (L = 4)
  void* y;        // [T, H] same type
  int residual;   // 1: y = x + MoE(x)
  int act_f32;    // 1: x and y are fp32 (check mode), else bf16
  int out_f32;    // 1: y is fp32 whatever the act dtype (moe_forward_f32)
  // residual-stream mode (moe_forward_resnorm), when h_in is set: y is not
  // written; h_out = h_in + MoE(x) in fp32 and xn = rmsnorm(h_out) in the act
  // dtype (weight 1, eps); ssq [8][n_dt] holds each block's per-token sum of
  // squares
  const float* h_in;
  float* h_out;
  void* xn;
  float eps;
  float* ssq;
  // workspace
  Sync* sync;
  int* status;
  unsigned long long* stamps;  // [2][kNumStamps]: this launch, then the last completed launch
  int* gu_cnt;       // [w_max]
  int* entry_ready;  // [w_max]
  int* d_cnt;        // [n_dt]
  long long* lfx;    // [E_pad][8] router logits in units of 2^-32, summed with integer atomics from the bias
                     // (restored to the bias by the routing block once it has read them)
  const long long* lfx0;  // [E_pad] the bias in units of 2^-32 (0 past E or without a bias): lfx's start
  int* ids;          // [T*k]
  float* gates;      // [T*k]
  int* pos;          // [T*k]
  int* offsets;      // [E+1]
  int* perm;         // [T*k]
  Entry* entries;    // [w_max]
  uint8_t* xrec;     // [T][H/32] records
  uint8_t* hrec;     // [P][Imax/32] records
  float* z;          // [P][H]
  // shared-memory plan
  int n_stages, ring_bytes, misc_bytes;  // descriptor slots, bytes of the stage ring, router scratch
  uint64_t timeout_ns;
  int ready_target;  // value of routing_ready the producers wait for: 1 (2^30 only under moe_layer_inject_timeout)
};

}  // namespace moe

struct moe_layer {
  int dev = 0;
  int H = 0, E = 0, k = 0, I = 0, Ish = 0, T_max = 0, act = 0;
  int e0 = 0, n_e = 0;          // routed experts held: [e0, e0 + n_e) of the E the router scores
  uint64_t timeout_ns = 0;      // bound of every device-side wait
  int inject = 0;               // one-shot wait-timeout test hook (moe_layer_inject_timeout)
  int fmt = 0, sfmt = 0;
  uint8_t* router = nullptr;
  float* router_b = nullptr;
  uint8_t* gu = nullptr;
  uint8_t* dn = nullptr;
  uint8_t* sgu = nullptr;
  uint8_t* sdn = nullptr;
  int64_t gu_stride = 0, dn_stride = 0;
  moe::Chunking gu_ch{}, dn_ch{}, sgu_ch{}, sdn_ch{};
  size_t weight_bytes = 0;
  // small-T workspace
  void* ws = nullptr;
  size_t ws_bytes = 0;
  moe::SmallParams sp{};  // pointers filled at create; T-dependent fields per call
  int num_sms = 0;
  int smem_bytes = 0;
  int last_T = 0;
  // prefill-sized path (T > kMaxSmallT), present when T_max > kMaxSmallT
  moe::LtState* lt = nullptr;
};

// Output norm + LM head of the MTP round (lm_head.cu, mtp.cu).
struct moe_lm_head {
  int dev = 0, V = 0, H = 0, T_max = 0, act = 0, num_sms = 0, max_optin = 0;
  uint8_t* w = nullptr;  // [ceil(V/32)][nch][Q8_0 chunk of 32 rows]
  int* status = nullptr; // [4]: timeout flag and wait site
};

namespace moe {
// Records a formatted message for moe_last_error() and returns `code` (api.cu).
int set_error(int code, const char* fmt, ...);
}  // namespace moe
