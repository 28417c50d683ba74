// verify.cu -- the two kernels of one verification call.
//
// plan_kernel (1 CTA): takes the call's epoch from the device-wide call
// counter, resets the counters, settles the requests whose inputs are
// invalid up front, and writes the position-major row schedule.
//
// verify_kernel: a persistent, warp-specialised kernel (every CTA resident,
// 2 per SM) that takes a request from its logits to its committed tokens.
// Work items come from three queues: the static schedule of 64 KB chunks of
// logit rows, the deferred queue (draft rows needed for the signals only,
// read after the static queue), and the draw queue created on the fly:
//   IT_STATS   softmax statistics of one chunk of a row (max m, s = sum
//              2^{(x-m)c}, for signal rows t = sum (x-m)c 2^{(x-m)c}, greedy
//              rows the max and its lowest index);
//   IT_DSUM    the weights of the final draw over one 16 KB slice of row k:
//              the residual [p_k - q_k]_+ (reject, full q: rows k of both
//              models) or p_k (bonus draw; one-hot reject with y_k removed);
//              fp32 sums per 256-token group and the fp64 slice sum are kept
//              (tutorial page "5.1 投机解码核心原理", sections 3.2, 3.3, 5.2).
// Roles inside a CTA:
//   producer (1 thread)  claims items, skips rows an earlier reject voided
//                   (defers signal-only draft rows), stages the bytes into a
//                   6-deep ring of 16 KB shared-memory buffers with
//                   cp.async.bulk completed on mbarriers;
//   8 consumer warps  read the staged bytes with 128-bit shared loads and do
//                   the arithmetic of the item;
//   2 epilogue warps  merge each chunk's 8 warp partials and publish them as
//                   tagged words (see tword);
//   owner warp      serves requests b = CTA, CTA + grid, ...: merges their
//                   rows from the tagged partials in fixed order, reads the
//                   logits at the draft tokens itself, tests the positions in
//                   order (sections 3.1-3.3, 5.1), publishes the
//                   first reject (early exit), runs the draw and writes the
//                   outputs.  Every decision of a request is taken in one warp.
// Every spin is bounded; a wait that gives up sets SPEC_ST_TIMEOUT, the other
// roles then give up too, and the last CTA to leave voids any request left
// unfinished.
#include <climits>

#include "common.cuh"
#include "exp2_table.cuh"

namespace sv {
namespace {

constexpr int kVoidMask = ~(SPEC_ST_ZERO_RESIDUAL | SPEC_ST_GUARDED);
constexpr int kFinished = 1 << 30;                 // req_status: outputs written
// A fast (fp32) draw whose token lies within kDrawGuard W of an edge of its
// bucket is taken again in extended precision.  fp32 weights and row sums
// move a bucket edge by a few 1e-8 W (modelled on the kernel's roundings of
// the residual for the bench workloads: at most 5e-8 W with the scale carried
// as c + c_lo; a p draw has the same exponent and fewer roundings); the
// guard is three times that.
constexpr float kDrawGuard = 1.5e-7f;

__device__ __forceinline__ float qnan() { return __int_as_float(0x7fc00000); }

__device__ __forceinline__ int gamma_of(const Params& P, int b) { return P.gamma ? P.gamma[b] : P.G; }

// Outputs of a request that commits nothing (an error found up front or on
// the way); `st` holds the error bits.  Any number of threads, strided by n.
__device__ void write_void_outputs(const Params& P, int b, int st, int t, int n) {
  const int G = P.G;
  if (P.mode != MODE_SIGNALS) {
    for (int j = t; j <= G; j += n) P.tokens[(size_t)b * (G + 1) + j] = -1;
    if (P.accept_prob)
      for (int j = t; j < G; j += n) P.accept_prob[(size_t)b * G + j] = qnan();
    if (t == 0) P.accept_len[b] = 0;
  }
  if (P.signals && t == 0)
    for (int j = 0; j < 4; ++j) P.signals[(size_t)b * 4 + j] = qnan();
  if (P.row_signals)
    for (int j = t; j < 2 * G; j += n) P.row_signals[(size_t)b * 2 * G + j] = qnan();
  if (t == 0 && P.status) P.status[b] = st;
}

}  // namespace

// ---------------------------------------------------------------------------
// plan: reset the counters and build the compacted row schedule

namespace {

enum BlockType : int { BT_T = 0, BT_D = 1, BT_PAIR = 2 };

struct Block {
  int type, i;
};

// Static schedule blocks in position-major order.  PAIR(i) holds target
// row i and (full q) draft row i of every request, so the rows a position's
// test needs come together.  Positions below the lookahead are read up front
// (sample and one-hot calls: 0 and 1; greedy calls: all); the rows of a later
// position i are enqueued by the request's owner once position
// i - lookahead is accepted.  With the signals on, every draft row is needed,
// so the draft rows past the lookahead also follow as D(i) blocks: a chunk of
// such a row is read by whichever comes first, the static item or the
// owner's entry (the other finds it claimed).
__device__ inline int build_blocks(int mode, int signals_on, int G, int lookahead, Block* out) {
  int n = 0;
  if (mode == MODE_SIGNALS) {
    for (int i = 0; i < G; ++i) out[n++] = {BT_D, i};
  } else if (mode == MODE_SAMPLE) {
    for (int i = 0; i <= G && i < lookahead; ++i) out[n++] = {BT_PAIR, i};
    if (signals_on)
      for (int i = lookahead; i < G; ++i) out[n++] = {BT_D, i};
  } else {
    for (int i = 0; i <= G && i < lookahead; ++i) out[n++] = {BT_T, i};
  }
  return n;
}

__device__ inline int rows_for(const Block& bl, int gam) {
  const int nt = gam >= bl.i ? 1 : 0;
  const int nd = gam > bl.i ? 1 : 0;
  if (bl.type == BT_T) return nt;
  if (bl.type == BT_D) return nd;
  return nt + nd;
}

}  // namespace

// Words of the tagged arrays, for the one-time clear of a new workspace.
__device__ inline void clear_tagged(const Params& P, int tid, int nth) {
  const size_t n_parts = (size_t)P.nrows * P.nch * kPartWords;
  const size_t n_dsum = (size_t)kSliceWords * P.B * P.nres;
  const size_t n_gsum = (size_t)P.B * P.nres * kGroupsPerStage * kGroupWords;
  for (size_t j = tid; j < n_parts; j += nth) P.cparts[j] = 0ull;
  for (size_t j = tid; j < n_dsum; j += nth) P.dsum[j] = 0ull;
  for (size_t j = tid; j < n_gsum; j += nth) P.gsum[j] = 0ull;
  for (size_t j = tid; j < (size_t)kDrawWords * P.B; j += nth) P.dd[j] = 0ull;
  for (size_t j = tid; j < 2 * (size_t)P.dq_cap; j += nth) P.dq[j] = 0ull;
  for (size_t j = tid; j < (size_t)P.B * P.G * P.nch; j += nth) P.claim[j] = 0ull;
  for (size_t j = tid; j < (size_t)P.def_cap; j += nth) P.defq[j] = 0ull;
}

// Calls of the plan kernel on this device so far (the source of every epoch).
__device__ unsigned long long g_calls = 0ull;

__global__ void __launch_bounds__(1024) plan_kernel(const __grid_constant__ Params P) {
  griddep_launch();
  const int B = P.B, G = P.G, tid = threadIdx.x, nth = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nth >> 5;
  __shared__ int s_count[64];
  __shared__ int s_off[65];
  __shared__ Block s_blk[64];
  __shared__ int s_nb;
  __shared__ unsigned s_settled;
  __shared__ unsigned s_epoch;
  __shared__ unsigned long long s_gen;
  __shared__ int s_clear;
  // gamma of each request whose rows are read (-1: none), for the row loops
  // below (calls with more requests read req_flags and gamma again)
  constexpr int kPlanB = 4096;
  __shared__ int s_gam[kPlanB];
  const bool small = B <= kPlanB;

  // The epoch of this call comes from one counter of calls on the device,
  // shared by every workspace: no two calls of a generation (kEpochMax - 1
  // calls) have the same epoch, so a word left in memory by any earlier call,
  // in this workspace or in another one that held the same memory, never
  // carries a tag of this call.  A workspace without the magic word (first
  // use), last cleared in another generation or last used by another copy
  // of this code (another counter) has its tagged arrays cleared (tag 0 is
  // never used).
  // (taken while the requests are checked below)
  unsigned long long n_calls = 0ull, hdr_magic = 0ull, hdr_gen = 0ull, hdr_owner = 0ull;
  if (tid == 0) {
    s_settled = 0u;
    n_calls = atomicAdd(&g_calls, 1ull);
    hdr_magic = HDR_MAGIC(P.hdr);
    hdr_gen = HDR_GEN(P.hdr);
    hdr_owner = HDR_OWNER(P.hdr);
  }
  __syncthreads();   // s_settled
  for (int b = tid; b < B; b += nth) {
    P.known_reject[b] = kNoReject;
    int st = 0;
    const int gam = gamma_of(P, b);
    if (gam < 0 || gam > G) st |= SPEC_ST_BAD_GAMMA;
    if (P.mode != MODE_GREEDY && !temperature_ok(P.temperature[b])) st |= SPEC_ST_BAD_TEMPERATURE;
    P.req_flags[b] = st;
    P.req_gam[b] = gam;
    P.req_scale[b] = (P.mode != MODE_GREEDY && st == 0) ? scale_of(P.temperature[b]) : 0.f;
    // the remainder (>= 0) of log2(e) / T past its fp32 value: the scale is
    // carried as hi + lo everywhere (see ref_of)
    P.req_scale_lo[b] = (P.mode != MODE_GREEDY && st == 0)
                            ? (float)(1.4426950408889634 / (double)P.temperature[b] - (double)P.req_scale[b])
                            : 0.f;
    P.req_ks[b] = scale_k(P.req_scale[b], P.req_scale_lo[b]);
    if (st != 0) {
      write_void_outputs(P, b, st, 0, 1);
      P.req_status[b] = st | kFinished;
      atomicAdd(&s_settled, 1u);
    } else if (P.mode == MODE_SIGNALS && gam == 0) {
      write_void_outputs(P, b, 0, 0, 1);      // signals of an empty draft are NaN
      P.req_status[b] = kFinished;
      atomicAdd(&s_settled, 1u);
    } else {
      P.req_status[b] = 0;
    }
    if (small) s_gam[b] = st == 0 ? gam : -1;
  }
  if (tid == 0) {
    s_nb = build_blocks(P.mode, P.signals_on, G, P.lookahead, s_blk);
    const unsigned long long gen = n_calls / (kEpochMax - 1u);
    s_epoch = 1u + (unsigned)(n_calls % (kEpochMax - 1u));
    s_gen = gen;
    s_clear = !(hdr_magic == kWorkspaceMagic && hdr_gen == gen &&
                hdr_owner == (unsigned long long)(uintptr_t)&g_calls);
  }
  __syncthreads();   // req_flags, s_gam, the block table and the epoch visible to the whole block
  if (s_clear) clear_tagged(P, tid, nth);
  // gamma of request b if its rows are read, else -1
  auto eligible = [&](int b) -> int {
    if (small) return s_gam[b];
    return P.req_flags[b] == 0 ? gamma_of(P, b) : -1;
  };

  const int nb = s_nb;
  // rows per block
  for (int k = warp; k < nb; k += nwarps) {
    const Block bl = s_blk[k];
    int cnt = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      int n = 0;
      if (b < B) {
        const int g = eligible(b);
        if (g >= 0) n = rows_for(bl, g);
      }
      cnt += __reduce_add_sync(0xffffffffu, n);
    }
    if (lane == 0) s_count[k] = cnt;
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int k = 0; k < nb; ++k) { s_off[k] = acc; acc += s_count[k]; }
    s_off[nb] = acc;
    P.hdr->queue.v = 0u;
    HDR_EPOCH(P.hdr) = s_epoch;
    HDR_MAGIC(P.hdr) = kWorkspaceMagic;
    HDR_GEN(P.hdr) = s_gen;
    HDR_OWNER(P.hdr) = (unsigned long long)(uintptr_t)&g_calls;
    HDR_N_ITEMS(P.hdr) = (unsigned)acc * (unsigned)P.nch;
    int nfront = 0;          // blocks of the first positions (all but the signal-only D blocks)
    while (nfront < nb && !(s_blk[nfront].type == BT_D && P.mode == MODE_SAMPLE)) ++nfront;
    HDR_N_FRONT(P.hdr) = (unsigned)s_off[nfront] * (unsigned)P.nch;
    P.hdr->error.v = 0u;
    HDR_UNCERTAIN(P.hdr) = 0u;
    P.hdr->dq_head.v = 0u;
    P.hdr->dq_tail.v = 0u;
    P.hdr->def_head.v = 0u;
    P.hdr->def_tail.v = 0u;
    P.hdr->done.v = 0u;
    HDR_N_VALID(P.hdr) = (unsigned)B - s_settled;
    HDR_EXITED(P.hdr) = 0u;
  }
  __syncthreads();
  // write the compacted row ids
  for (int k = warp; k < nb; k += nwarps) {
    const Block bl = s_blk[k];
    int off = s_off[k];
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      int n = 0, gam = 0;
      if (b < B) {
        gam = eligible(b);
        if (gam >= 0) n = rows_for(bl, gam);
      }
      int incl = n;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, d);
        if (lane >= d) incl += v;
      }
      int pos = off + incl - n;
      if (n > 0) {
        const bool want_t = bl.type != BT_D && gam >= bl.i;
        const bool want_d = bl.type != BT_T && gam > bl.i;
        if (want_t) P.row_list[pos++] = target_row_id(b, bl.i, G);
        if (want_d) P.row_list[pos++] = draft_row_id(b, bl.i, B, G);
      }
      off += __shfl_sync(0xffffffffu, incl, 31);
    }
  }
}


// ---------------------------------------------------------------------------
// persistent kernel: shared state

namespace {

constexpr int F_FIRST = 1, F_LAST = 2, F_TERM = 4, F_DIRECT = 8, F_DRAW = 16;
constexpr int kItemSlots = 16;      // see ItemDesc

// One work item (producer -> consumers), written once, when its first stage
// is issued, into slot (item number mod kItemSlots).  A draw slice (one or
// two stages) may be issued between two stages of a statistics item (at most
// three times, one per stage boundary), so the stages of the kItemSlots - 1
// items issued after an item span at most 3 * 2 + kItemSlots - 1 stages past
// its first; the slot is written again only when the ring slot of item
// (n + kItemSlots)'s first stage is free, i.e. once every consumer warp has
// released the stage kStages before it, which lies past item n's last stage
// and its chunk-end work.  So consumers read item fields in shared memory
// when they need them and hold none in registers over a stage.
struct ItemDesc {
  int b, i, kind, row_id;
  int chunk, y, aux, head0;
  int nhead, tail0, ntail;
  float c, m1, s1, m2, s2;
  unsigned tag;                     // draw: tag of the draw's words
  float c_lo, r1h, r1l, r2h, r2l;   // extended-precision draws: scale remainder, 1/S_p, 1/S_q
  float ks;                         // statistics items: the exponent stretch (see ref_of)
  int pad[1];
};

// One staged piece of an item (producer -> consumers): 16 bytes.
struct StageDesc {
  int flags;                        // F_FIRST | F_LAST | F_TERM | F_DIRECT | F_DRAW
  int nvec;                         // 16-byte vectors in the stage
  int elem0;                        // row element of the stage's first element
  int item;                         // item slot | row kind << 4 (draw slices: target, then draft)
};

// One finished item (consumers -> epilogue).
struct EpiSlot {
  int type, row_id, b, i;
  int kind, chunk, term, z;
  unsigned tag;                     // draw: tag of the draw's words
  float c, ks;                      // statistics: the request's scale and stretch
  int pad[1];
  double dsum[kConsumerWarps];      // draw-weight sums per consumer warp (IT_DSUM)
  double dsum2[kConsumerWarps];     // second sum (S_q) of a DK_SUMS slice
  Part part[kConsumerWarps];        // statistics per consumer warp (IT_STATS)
};

// One unit of work handed from the scheduler to the producer (shared
// memory): a row chunk with its request's values, a draw slice with its
// round's descriptor words, or the end.
enum WorkType : int { WT_ROW = 1, WT_DRAW = 2, WT_TERM = 3 };
struct WorkEntry {
  int type;
  int rid, chunk;                   // WT_ROW: row id, chunk; WT_DRAW: request b, slice
  float c, ks;                      // WT_ROW: the request's scale and stretch
  unsigned tag;                     // WT_DRAW: the round's tag
  int urgent;                       // WT_DRAW: a round after the first (a retake)
  unsigned v[kDrawWords];           // WT_DRAW: the round's descriptor words
};
constexpr int kFifo = 1;            // row chunks handed over ahead of the producer (claimed late: a decided reject skips more)

struct __align__(128) VSmem {
  unsigned char ring[kStages][kStageBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t epi_full[kEpiSlots];
  uint64_t epi_empty[kEpiSlots];
  StageDesc desc[kStages];
  ItemDesc item[kItemSlots];
  EpiSlot slot[kEpiSlots];
  float2 exp2tab[256];              // 2^{i/256} as hi, lo (extended-precision draws)
  WorkEntry fifo[kFifo];            // scheduler -> producer: row chunks (and the end marker)
  WorkEntry prio;                   // scheduler -> producer: one draw slice
  int fifo_head, fifo_tail, prio_full;
  long long wait_limit;             // Params::wait_limit, for the waits that see only S
  int abort;
};

}  // namespace

namespace {

__device__ __forceinline__ bool aborted(const VSmem& S) {
  return *reinterpret_cast<const volatile int*>(&S.abort) != 0;
}

__device__ __forceinline__ void set_abort(const Params& P, VSmem& S) {
  *reinterpret_cast<volatile int*>(&S.abort) = 1;
  atomicOr(&P.hdr->error.v, (unsigned)SPEC_ST_TIMEOUT);
}

// Bounded wait that also gives up when another role of the CTA aborted.
// The wait sleeps in hardware between checks (at most kSleepHintNs each).
constexpr uint32_t kSleepHintNs = 100000;
__device__ __forceinline__ bool wait_bar(VSmem& S, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long c0 = clock64();
  while (true) {
    if (mbar_try_wait_sleep(bar, parity, kSleepHintNs)) return true;
    if (aborted(S)) return false;
    if (clock64() - c0 > S.wait_limit) return false;
  }
}

template <int DT>
struct VecT;
template <>
struct VecT<SPEC_BF16> {
  static constexpr int N = 8;
  __device__ static __forceinline__ void unpack(const uint4& w, float* x) {
    x[0] = bf16_lo(w.x); x[1] = bf16_hi(w.x); x[2] = bf16_lo(w.y); x[3] = bf16_hi(w.y);
    x[4] = bf16_lo(w.z); x[5] = bf16_hi(w.z); x[6] = bf16_lo(w.w); x[7] = bf16_hi(w.w);
  }
};
template <>
struct VecT<SPEC_F32> {
  static constexpr int N = 4;
  __device__ static __forceinline__ void unpack(const uint4& w, float* x) {
    x[0] = __uint_as_float(w.x); x[1] = __uint_as_float(w.y);
    x[2] = __uint_as_float(w.z); x[3] = __uint_as_float(w.w);
  }
};

// Per-thread running state of one chunk.
struct RunState {
  float m, s, t, mc;
  int idx;
  int nan;
};

__device__ __forceinline__ void run_reset(RunState& r) {
  r.m = -INFINITY; r.s = 0.f; r.t = 0.f; r.mc = 0.f; r.idx = 0x3fffffff; r.nan = 0;
}

// ---- per-stage processing ---------------------------------------------------
// Each consumer thread owns 4 of the stage's 1024 16-byte vectors (strided by
// 256, so every shared load of a warp is one contiguous 512-byte run).  The
// stage max is taken first with a max tree (one running-max update per stage,
// not per vector), then the 32 (bf16) or 16 (fp32) terms are independent, so
// their exp2 and adds pipeline.  Vectors past the staged bytes read as -inf.

constexpr int kVecPerThread = kStageBytes / 16 / kConsumerThreads;   // 4
static_assert(kVecPerThread == 4, "the draw's group sums take four vectors per thread");

__device__ __forceinline__ uint32_t bmax2(uint32_t a, uint32_t b) {       // NaN-ignoring
  uint32_t d;
  asm("max.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
__device__ __forceinline__ uint32_t bmax2_nan(uint32_t a, uint32_t b) {   // NaN-propagating
  uint32_t d;
  asm("max.NaN.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}

template <int DT>
__device__ __forceinline__ void load_stage(const uint4* vec, int nvec, int tid, uint4 (&w)[kVecPerThread]) {
  if (nvec == kStageBytes / 16) {     // a full stage (all but a row's last)
#pragma unroll
    for (int r = 0; r < kVecPerThread; ++r) w[r] = vec[tid + r * kConsumerThreads];
    return;
  }
  const uint32_t ninf = DT == SPEC_BF16 ? 0xff80ff80u : 0xff800000u;
#pragma unroll
  for (int r = 0; r < kVecPerThread; ++r) {
    const int v = tid + r * kConsumerThreads;
    w[r] = v < nvec ? vec[v] : make_uint4(ninf, ninf, ninf, ninf);
  }
}

// max over the thread's stage elements (NaN ignored or propagated)
template <int DT, bool NANP>
__device__ __forceinline__ float stage_max(const uint4 (&w)[kVecPerThread]) {
  if (DT == SPEC_BF16) {
    uint32_t h[2 * kVecPerThread];
#pragma unroll
    for (int r = 0; r < kVecPerThread; ++r) {
      h[2 * r] = NANP ? bmax2_nan(w[r].x, w[r].y) : bmax2(w[r].x, w[r].y);
      h[2 * r + 1] = NANP ? bmax2_nan(w[r].z, w[r].w) : bmax2(w[r].z, w[r].w);
    }
#pragma unroll
    for (int n = 2 * kVecPerThread; n > 1; n >>= 1)
#pragma unroll
      for (int k = 0; k < n / 2; ++k) h[k] = NANP ? bmax2_nan(h[2 * k], h[2 * k + 1]) : bmax2(h[2 * k], h[2 * k + 1]);
    const float lo = bf16_lo(h[0]), hi = bf16_hi(h[0]);
    if (NANP && (lo != lo || hi != hi)) return __int_as_float(0x7fc00000);
    return fmaxf(lo, hi);
  } else {
    float f[4 * kVecPerThread];
#pragma unroll
    for (int r = 0; r < kVecPerThread; ++r) {
      f[4 * r] = __uint_as_float(w[r].x); f[4 * r + 1] = __uint_as_float(w[r].y);
      f[4 * r + 2] = __uint_as_float(w[r].z); f[4 * r + 3] = __uint_as_float(w[r].w);
    }
    bool nan = false;
    if (NANP) {
#pragma unroll
      for (int k = 0; k < 4 * kVecPerThread; ++k) nan |= f[k] != f[k];
    }
#pragma unroll
    for (int n = 4 * kVecPerThread; n > 1; n >>= 1)
#pragma unroll
      for (int k = 0; k < n / 2; ++k) f[k] = fmaxf(f[2 * k], f[2 * k + 1]);
    return nan ? __int_as_float(0x7fc00000) : f[0];
  }
}

// -inf logits must contribute 0 to t = sum a 2^a, not -inf * 0.  For bf16
// signal rows the staged words are clamped at -2^100 with one packed max per
// two logits (the stage max is taken before, on the raw words, so a row of
// -inf still has no finite max); 2^{-2^100 c} is 0 and its product with the
// finite exponent is 0.  For fp32 rows, or scales large enough that the
// clamped exponent could overflow, the exponent itself is clamped.
constexpr uint32_t kClampWords = 0xF180F180u;   // bf16 pair (-2^100, -2^100)
constexpr float kClampScaleMax = 1048576.f;

// Packed fp32 pairs (Blackwell FFMA2 / FADD2): the exponent, the sum tree
// and the entropy product run two logits per instruction.
__device__ __forceinline__ float2 f2(float a, float b) { return make_float2(a, b); }

template <int DT, bool ENT>
__device__ __forceinline__ void stage_softmax(RunState& r, uint4 (&w)[kVecPerThread], float c, float ks) {
  using Vec = VecT<DT>;
  constexpr int N = Vec::N;
  constexpr int NP = N / 2;                     // pairs per vector
  const float vm = stage_max<DT, false>(w);
  if (vm > r.m) {
    const float vmc = ref_of(vm, c);
    if (r.m != -INFINITY) {
      const float d = stretch(__fsub_rn(r.mc, vmc), ks);
      const float f = ex2(d);
      if (ENT) r.t = f * fmaf(d, r.s, r.t);
      r.s *= f;
    }
    r.m = vm;
    r.mc = vmc;
  }
  const bool packed_clamp = ENT && DT == SPEC_BF16 && c <= kClampScaleMax;
  if (packed_clamp) {
#pragma unroll
    for (int q = 0; q < kVecPerThread; ++q) {
      w[q].x = bmax2_nan(w[q].x, kClampWords); w[q].y = bmax2_nan(w[q].y, kClampWords);
      w[q].z = bmax2_nan(w[q].z, kClampWords); w[q].w = bmax2_nan(w[q].w, kClampWords);
    }
  }
  const float2 C2 = f2(c, c), K2 = f2(ks, ks), NMC2 = f2(-r.mc, -r.mc), LO2 = f2(-256.f, -256.f);
  float2 s2 = f2(0.f, 0.f), t2 = f2(0.f, 0.f);
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) {
    float x[N];
    Vec::unpack(w[q], x);
    float2 e[NP];
#pragma unroll
    for (int k = 0; k < NP; ++k) {
      float2 a = __ffma2_rn(f2(x[2 * k], x[2 * k + 1]), C2, NMC2);
      a = __ffma2_rn(a, K2, a);                    // stretch: the scale's remainder (see ref_of)
      e[k] = f2(ex2(a.x), ex2(a.y));
      if (ENT) {
        if (!packed_clamp) a = f2(fmaxf(a.x, LO2.x), fmaxf(a.y, LO2.y));
        t2 = __ffma2_rn(a, e[k], t2);
      }
    }
    float2 v;
    if (NP == 4) v = __fadd2_rn(__fadd2_rn(e[0], e[1]), __fadd2_rn(e[2], e[3]));
    else v = __fadd2_rn(e[0], e[1]);
    s2 = __fadd2_rn(s2, v);
  }
  r.s += s2.x + s2.y;
  if (ENT) r.t += t2.x + t2.y;
}

// Warp partial of a softmax run: the warp max first, one rescale of each
// lane's sums to it, then plain sums (fixed xor tree: deterministic).
__device__ __forceinline__ Part warp_softmax_part(const RunState& r, float c, float ks, bool ent) {
  float m = r.m;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float s = 0.f, t = 0.f;
  if (r.s != 0.f) {                       // lanes that saw nothing contribute 0
    const float d = stretch(__fsub_rn(r.mc, ref_of(m, c)), ks);
    const float f = ex2(d);
    s = r.s * f;
    if (ent) t = f * fmaf(d, r.s, r.t);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    s += __shfl_xor_sync(0xffffffffu, s, off);
    if (ent) t += __shfl_xor_sync(0xffffffffu, t, off);
  }
  Part p;
  p.m = m; p.s = s; p.t = t; p.idx = 0x3fffffff;
  return p;
}

template <int DT>
__device__ __forceinline__ void stage_argmax(RunState& r, const uint4 (&w)[kVecPerThread], int elem0, int tid) {
  using Vec = VecT<DT>;
  constexpr int N = Vec::N;
  const float vm = stage_max<DT, true>(w);
  if (vm != vm) { r.nan = 1; return; }
  if (vm > r.m) {
    int idx = 0x3fffffff;
#pragma unroll
    for (int q = kVecPerThread - 1; q >= 0; --q) {
      float x[N];
      Vec::unpack(w[q], x);
#pragma unroll
      for (int k = N - 1; k >= 0; --k)
        if (x[k] == vm) idx = elem0 + (tid + q * kConsumerThreads) * N + k;
    }
    r.m = vm;
    r.idx = idx;
  }
}

// one scalar logit at row element `e` (head/tail of a chunk)
template <bool GREEDY>
__device__ __forceinline__ void run_scalar(RunState& r, float x, int e, float c, float ks, bool ent) {
  if (GREEDY) {
    r.nan |= x != x;
    if (x > r.m || (x == r.m && e < r.idx)) { r.m = x; r.idx = e; }
    return;
  }
  if (x > r.m) {
    const float xc = ref_of(x, c);
    if (r.m != -INFINITY) {
      const float d = stretch(__fsub_rn(r.mc, xc), ks);
      const float f = ex2(d);
      if (ent) r.t = f * fmaf(d, r.s, r.t);
      r.s *= f;
    }
    r.m = x;
    r.mc = xc;
  }
  const float a = stretch(fmaf(x, c, -r.mc), ks);
  const float ev = ex2(a);
  r.s += ev;
  if (ent) r.t = fmaf(fmaxf(a, -256.f), ev, r.t);
}

__device__ __forceinline__ Part to_part(const RunState& r) {
  Part p;
  p.m = r.m; p.s = r.s; p.t = r.t;
  p.idx = (r.idx & ~kIdxNaN) | (r.nan ? kIdxNaN : 0);
  return p;
}


// ---------------------------------------------------------------------------
// small memory-model helpers

__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// ---------------------------------------------------------------------------
// device work queue

// Tags of this call's words (see tword).
__device__ __forceinline__ unsigned draw_tag(unsigned epoch, int round) { return (8u * epoch + 1u + (unsigned)round) * kTagMul; }
__device__ __forceinline__ unsigned part_tag(unsigned epoch) { return 8u * epoch * kTagMul; }   // partials, queue entries

// An entry is two tagged words: (b) and (slice | round << 30), both with the
// call's partial tag.  The owner of request b reserves n consecutive entries
// (slices 0 .. n-1) and every lane of its warp writes entries lane,
// lane + 32, ...  Warp-wide.
__device__ __forceinline__ void enqueue_draw(const Params& P, int n, int b, int round, unsigned epoch, int lane) {
  unsigned base = 0;
  if (lane == 0) base = atomicAdd(&P.hdr->dq_tail.v, (unsigned)n);
  base = __shfl_sync(0xffffffffu, base, 0);
  for (int j = lane; j < n; j += 32) {
    const unsigned slot = base + (unsigned)j;
    if (slot >= (unsigned)P.dq_cap) {       // cannot happen; keeps every write in bounds
      atomicOr(&P.hdr->error.v, (unsigned)SPEC_ST_TIMEOUT);
      continue;
    }
    st_tw(P.dq + 2 * (size_t)slot, tw_make((unsigned)b, part_tag(epoch)));
    st_tw(P.dq + 2 * (size_t)slot + 1, tw_make((unsigned)j | ((unsigned)round << 30), part_tag(epoch)));
  }
  __syncwarp();
}

// Lookahead rows: the owner enqueues every chunk of row rid (entries
// (rid | 1 << 31), chunk).  Warp-wide.
__device__ __forceinline__ void enqueue_row(const Params& P, int rid, unsigned epoch, int lane) {
  unsigned base = 0;
  if (lane == 0) base = atomicAdd(&P.hdr->dq_tail.v, (unsigned)P.nch);
  base = __shfl_sync(0xffffffffu, base, 0);
  for (int j = lane; j < P.nch; j += 32) {
    const unsigned slot = base + (unsigned)j;
    if (slot >= (unsigned)P.dq_cap) {       // cannot happen; keeps every write in bounds
      atomicOr(&P.hdr->error.v, (unsigned)SPEC_ST_TIMEOUT);
      continue;
    }
    st_tw(P.dq + 2 * (size_t)slot, tw_make((unsigned)rid | 0x80000000u, part_tag(epoch)));
    st_tw(P.dq + 2 * (size_t)slot + 1, tw_make((unsigned)j, part_tag(epoch)));
  }
  __syncwarp();
}

// Dynamic items (draw slices and lookahead row chunks) are handed out by
// ticket: a producer holds one ticket (an index into the queue, from one
// atomicAdd) and takes the item stored there once both of its words carry
// this call's tag.  Tickets past the last item are never served; their
// holders leave when every request is done.


// The draw descriptor of request b (owner -> producers), kDrawWords tagged
// words: kind | k << 8, excluded token (one-hot), m_p, s_p, m_q, s_q, the
// scale and its remainder, 1 / S_p and 1 / S_q as hi, lo (DK_PRESID).
enum DrawWord : int {
  DW_KIND = 0, DW_EXCL, DW_M1, DW_S1, DW_M2, DW_S2, DW_C, DW_CLO, DW_R1H, DW_R1L, DW_R2H, DW_R2L, DW_END
};
static_assert(DW_END == kDrawWords, "draw descriptor size");


// ---------------------------------------------------------------------------
// producer

// A row chunk to stage: the row, the chunk, the request's scale and stretch.
struct RowItem {
  int rid, chunk;
  float c, ks;
};

// Stage one piece: wait for a free ring slot, let `fill` write the item's
// descriptor (the first piece of an item) into its slot, write the stage's,
// start the bulk copy (bytes > 0) or just mark the stage full.
template <class Fill>
__device__ __forceinline__ bool put_stage(VSmem& S, int& stage, uint32_t& phase, const StageDesc& d, bool first,
                                          Fill&& fill, uintptr_t src, uint32_t bytes, uint64_t policy) {
  if (!wait_bar(S, &S.empty[stage], phase ^ 1u)) return false;
  if (first) fill(S.item[d.item & (kItemSlots - 1)]);
  S.desc[stage] = d;
  if (bytes > 0) {
    mbar_arrive_expect_tx(&S.full[stage], bytes);
    bulk_load_hint(S.ring[stage], reinterpret_cast<const void*>(src), bytes, &S.full[stage], policy);
  } else {
    mbar_arrive(&S.full[stage]);
  }
  if (++stage == kStages) { stage = 0; phase ^= 1u; }
  return true;
}

// Draft-row chunks past the lookahead can be reached twice (a static item
// and an owner's lookahead entry): the first to swap the call's tag into the
// chunk's claim word reads it, the other skips it (before taking an item
// slot: every item number has at least one stage, see ItemDesc).
__device__ __forceinline__ bool claim_chunk(const Params& P, int kind, int b, int i, int chunk, unsigned ptag) {
  if (kind != KIND_DRAFT || i < P.lookahead || P.mode != MODE_SAMPLE) return true;
  const tword mine = tw_make(1u, ptag);
  const tword old = atomicExch(P.claim + ((size_t)b * P.G + i) * P.nch + chunk, mine);
  return old != mine;
}

// One chunk of a row, in bulk-copied pieces of up to one stage (aligned
// middle) plus scalar head/tail elements the consumers read themselves;
// `between` runs after each piece (the producer's work between stages).
template <int DT, bool GREEDY, class Hook>
__device__ __forceinline__ bool stage_row_item(const Params& P, VSmem& S, int& stage, uint32_t& phase, const RowItem& r, int islot,
                               Hook&& between) {
  constexpr int ES = DT == SPEC_BF16 ? 2 : 4;
  const int G = P.G, V = P.V;
  int kind, b, i;
  decode_row(r.rid, P.B, G, kind, b, i);
  const int ce = chunk_elems(DT);
  const unsigned char* tens = kind == KIND_TARGET ? P.target : P.draft;
  const long long row0 = row_elem_offset(kind, b, i, G, V);
  const int e_begin = r.chunk * ce;
  const int e_end = min(e_begin + ce, V);
  const uintptr_t rowaddr = reinterpret_cast<uintptr_t>(tens) + (uintptr_t)(row0 * ES);
  const uintptr_t a_start = rowaddr + (uintptr_t)e_begin * ES;
  const uintptr_t a_end = rowaddr + (uintptr_t)e_end * ES;
  uintptr_t A0 = (a_start + 15) & ~uintptr_t(15);
  uintptr_t A1 = a_end & ~uintptr_t(15);
  int nhead, ntail;
  if (A1 <= A0) {            // no aligned middle: everything is scalar head
    A0 = A1 = a_end;
    nhead = e_end - e_begin;
    ntail = 0;
  } else {
    nhead = (int)((A0 - a_start) / ES);
    ntail = (int)((a_end - A1) / ES);
  }
  const long long mid = (long long)(A1 - A0);
  const int npieces = mid > 0 ? (int)((mid + kStageBytes - 1) / kStageBytes) : 1;
  auto fill = [&](ItemDesc& D) {
    D.row_id = r.rid; D.b = b; D.i = i; D.kind = kind; D.chunk = r.chunk;
    D.head0 = e_begin; D.nhead = nhead; D.tail0 = e_end - ntail; D.ntail = ntail;
    D.c = r.c; D.ks = r.ks;
  };
  StageDesc d;
  d.item = islot;
  const uint64_t pol = l2_policy(i <= P.keep_pos);
  for (int p = 0; p < npieces; ++p) {
    const long long off = (long long)p * kStageBytes;
    const uint32_t bytes = mid > 0 ? (uint32_t)(mid - off < kStageBytes ? mid - off : kStageBytes) : 0u;
    d.elem0 = (int)((A0 + (uintptr_t)off - rowaddr) / ES);
    d.nvec = (int)(bytes / 16);
    d.flags = (p == 0 ? F_FIRST : 0) | (p == npieces - 1 ? F_LAST : 0);
    if (!put_stage(S, stage, phase, d, p == 0, fill, A0 + (uintptr_t)off, bytes, pol)) return false;
    between();
  }
  return true;
}

// Stage the elements [e0, e1) of one row (at most one stage worth) with a
// bulk copy when rows are 16-byte aligned, else as a direct stage that the
// consumers fill themselves.
template <int DT, class Fill>
__device__ __forceinline__ bool put_row_range(const Params& P, VSmem& S, int& stage, uint32_t& phase,
                                              StageDesc d, bool first, Fill&& fill, int kind, int b, int i, int e0,
                                              int e1) {
  constexpr int ES = DT == SPEC_BF16 ? 2 : 4;
  const unsigned char* tens = kind == KIND_TARGET ? P.target : P.draft;
  const long long src = row_elem_offset(kind, b, i, P.G, P.V) + e0;
  d.elem0 = e0;
  d.item = (d.item & (kItemSlots - 1)) | (kind << 4);
  if (P.aligned_rows) {
    const uint32_t bytes = (uint32_t)((e1 - e0) * ES);
    d.nvec = (int)(bytes / 16);
    return put_stage(S, stage, phase, d, first, fill, reinterpret_cast<uintptr_t>(tens) + (uintptr_t)(src * ES),
                     bytes, l2_policy(false));
  }
  d.flags |= F_DIRECT;
  d.nvec = (e1 - e0 + (16 / ES) - 1) / (16 / ES);
  return put_stage(S, stage, phase, d, first, fill, 0, 0u, 0ull);
}

// A draw slice from the priority slot: rows k of request b (one stage, or a
// target and a draft stage for a residual), with the round's descriptor
// words as the scheduler read them.
template <int DT>
__device__ __forceinline__ bool stage_draw_entry(const Params& P, VSmem& S, int& stage, uint32_t& phase,
                                                 const WorkEntry& e, int islot) {
  const int V = P.V, se = stage_elems(DT);
  const int b = e.rid, slice = e.chunk;
  const unsigned* v = e.v;
  const int kind = (int)(v[DW_KIND] & 0xffu), k = (int)(v[DW_KIND] >> 8);
  auto fill = [&](ItemDesc& D) {
    D.b = b; D.i = k; D.chunk = slice; D.aux = kind; D.y = (int)v[DW_EXCL]; D.tag = e.tag;
    D.c = __uint_as_float(v[DW_C]); D.c_lo = __uint_as_float(v[DW_CLO]);
    D.m1 = __uint_as_float(v[DW_M1]); D.s1 = __uint_as_float(v[DW_S1]);
    D.m2 = __uint_as_float(v[DW_M2]); D.s2 = __uint_as_float(v[DW_S2]);
    D.r1h = __uint_as_float(v[DW_R1H]); D.r1l = __uint_as_float(v[DW_R1L]);
    D.r2h = __uint_as_float(v[DW_R2H]); D.r2l = __uint_as_float(v[DW_R2L]);
  };
  const int e0 = slice * se, e1 = min(e0 + se, V);
  StageDesc d;
  d.item = islot;
  if (kind != DK_P && kind != DK_PF) {   // both rows k: target stage, then draft stage
    d.flags = F_DRAW | F_FIRST;
    if (!put_row_range<DT>(P, S, stage, phase, d, true, fill, KIND_TARGET, b, k, e0, e1)) return false;
    d.flags = F_DRAW | F_LAST;
    return put_row_range<DT>(P, S, stage, phase, d, false, fill, KIND_DRAFT, b, k, e0, e1);
  }
  d.flags = F_DRAW | F_FIRST | F_LAST;
  return put_row_range<DT>(P, S, stage, phase, d, true, fill, KIND_TARGET, b, k, e0, e1);
}

// The request values of a row item (two dependent loads after the row id)
template <bool GREEDY>
__device__ __forceinline__ void row_values(const Params& P, int rid, float& c, float& ks) {
  if (GREEDY) { c = ks = 0.f; return; }
  int kind, b, i;
  decode_row(rid, P.B, P.G, kind, b, i);
  c = __ldg(P.req_scale + b);
  ks = __ldg(P.req_ks + b);
}

__device__ __forceinline__ int ld_vol(const int* p) { return *reinterpret_cast<const volatile int*>(p); }
__device__ __forceinline__ void st_vol(int* p, int v) { *reinterpret_cast<volatile int*>(p) = v; }

// The producer (one thread) only moves bytes: it takes the work the
// scheduler hands over in shared memory (a FIFO of row chunks and a slot for
// one draw slice) and issues the bulk copies into the ring.  It never waits
// on global memory, so the ring stays full.  Draw slices and row chunks take
// turns: the rows of the positions still open are the longest chain of the
// call, while a draw started early has time to spare.  A retake round (a
// draw taken again near a tie) goes first, also between the stages of a row
// chunk: it is on the critical path of its request.
template <int DT, bool GREEDY>
__device__ __forceinline__ void producer_role(const Params& P, VSmem& S) {
  int stage = 0;
  uint32_t phase = 0;
  int islot = 0;              // items issued (their descriptor slots)
  bool ok = true;
  int head = 0;               // FIFO entries taken
  auto take_prio = [&]() {
    __threadfence_block();    // the entry as the scheduler wrote it
    ok = stage_draw_entry<DT>(P, S, stage, phase, S.prio, islot++ & (kItemSlots - 1));
    __threadfence_block();    // read before the slot is handed back
    st_vol(&S.prio_full, 0);
  };
  long long idle_since = -1;
  bool last_row = true;
  while (ok) {
    const bool rows = ld_vol(&S.fifo_tail) != head;
    if (ld_vol(&S.prio_full) && (last_row || !rows || ld_vol(&S.prio.urgent))) {
      take_prio();
      last_row = false;
      idle_since = -1;
      continue;
    }
    if (rows) {
      last_row = true;
      __threadfence_block();
      const WorkEntry& e = S.fifo[head % kFifo];
      if (e.type == WT_TERM) break;
      RowItem r;
      r.rid = e.rid; r.chunk = e.chunk; r.c = e.c; r.ks = e.ks;
      __threadfence_block();
      st_vol(&S.fifo_head, ++head);
      ok = stage_row_item<DT, GREEDY>(P, S, stage, phase, r, islot++ & (kItemSlots - 1), [&]() {
        if (ok && ld_vol(&S.prio_full) && ld_vol(&S.prio.urgent)) take_prio();
      });
      idle_since = -1;
      continue;
    }
    if (aborted(S)) { ok = false; break; }
    const long long now = clock64();
    if (idle_since < 0) idle_since = now;
    else if (now - idle_since > P.wait_limit) { ok = false; break; }
    __nanosleep(32);
  }
  if (ok && wait_bar(S, &S.empty[stage], phase ^ 1u)) {
    S.desc[stage].flags = F_TERM;
    mbar_arrive(&S.full[stage]);
    if (++stage == kStages) { stage = 0; phase ^= 1u; }
  } else {
    set_abort(P, S);                 // gave up: tell the other roles
  }
  // Let every copy this producer issued land before the CTA can exit: the
  // latest phase of each ring slot, always with the default limit (a copy of
  // valid memory completes; a consumer that gave up early under a lowered
  // limit may have left one in flight).
  for (int s = 0; s < kStages; ++s) {
    const uint32_t par = s < stage ? phase : phase ^ 1u;
    const long long c0 = clock64();
    while (!mbar_try_wait(&S.full[s], par) && clock64() - c0 < kWaitLimitCycles) {
    }
  }
}

// The scheduler (one thread) decides what the producer stages next.  It
// takes the work from global memory, where every step may wait on a load or
// an atomic: a dynamic entry at its ticket (a draw slice goes to the
// priority slot with its round's descriptor, a lookahead row chunk to the
// FIFO), else a static item (position-major main queue; a decided reject
// voids the row, and a draft row that only the signals still need goes to
// the deferred queue, shared by all CTAs, so the rows of live requests go
// first), else a deferred item.  It ends the producer with a WT_TERM entry
// once no work can come any more.
template <int DT, bool GREEDY>
__device__ __forceinline__ void scheduler_role(const Params& P, VSmem& S, unsigned epoch) {
  const unsigned n_items = HDR_N_ITEMS(P.hdr);
  const unsigned n_valid = HDR_N_VALID(P.hdr);
  const unsigned ptag = part_tag(epoch);
  // sample and one-hot calls have dynamic items: draw slices and lookahead rows
  const bool dyn = !GREEDY && (P.mode == MODE_SAMPLE || P.mode == MODE_ONEHOT);
  const bool defer_on = dyn && P.mode == MODE_SAMPLE && P.signals_on;
  unsigned ticket = dyn ? atomicAdd(&P.hdr->dq_head.v, 1u) : 0xffffffffu;
  bool main_done = n_items == 0u;
  unsigned dticket = 0xffffffffu;     // deferred-queue ticket whose entry is not seen yet
  int tail = 0;
  bool ok = true;
  auto room = [&]() { return tail - ld_vol(&S.fifo_head) < kFifo; };
  auto push = [&](int type, int rid, int chunk, float c, float ks) {
    WorkEntry& e = S.fifo[tail % kFifo];
    e.type = type; e.rid = rid; e.chunk = chunk; e.c = c; e.ks = ks;
    __threadfence_block();
    st_vol(&S.fifo_tail, ++tail);
  };
  auto push_row = [&](int rid, int chunk) {
    float c, ks;
    row_values<GREEDY>(P, rid, c, ks);
    push(WT_ROW, rid, chunk, c, ks);
  };
  long long idle_since = -1;
  unsigned sleep_ns = 32;
  while (ok) {
    bool did = false;
    // 1. the dynamic entry at the held ticket
    if (dyn && ticket < (unsigned)P.dq_cap) {
      const tword w0 = ld_tw(P.dq + 2 * (size_t)ticket), w1 = ld_tw(P.dq + 2 * (size_t)ticket + 1);
      if (tw_ok(w0, ptag) && tw_ok(w1, ptag)) {
        const unsigned e0 = tw_u32(w0), e1 = tw_u32(w1);
        if (e0 >> 31) {                       // a lookahead row chunk
          if (room()) {
            ticket = atomicAdd(&P.hdr->dq_head.v, 1u);
            const int rid = (int)(e0 & 0x7fffffffu), chunk = (int)e1;
            int kind, b, i;
            decode_row(rid, P.B, P.G, kind, b, i);
            if (claim_chunk(P, kind, b, i, chunk, ptag)) push_row(rid, chunk);
            did = true;
          }
        } else if (!ld_vol(&S.prio_full)) {   // a draw slice: its round's descriptor first
          const int b = (int)e0, slice = (int)(e1 & 0x3fffffffu), round = (int)(e1 >> 30);
          const unsigned tag = draw_tag(epoch, round);
          const tword* dd = P.dd + (size_t)b * kDrawWords;
          WorkEntry& e = S.prio;
          const long long c0 = clock64();
          while (true) {
            bool all = true;
#pragma unroll
            for (int j = 0; j < kDrawWords; ++j) {
              const tword w = ld_tw(dd + j);
              all &= tw_ok(w, tag);
              e.v[j] = tw_u32(w);
            }
            if (all) break;
            if (aborted(S) || clock64() - c0 > P.wait_limit) { ok = false; break; }
          }
          if (!ok) break;
          e.type = WT_DRAW; e.rid = b; e.chunk = slice; e.tag = tag; e.urgent = round > 0;
          __threadfence_block();
          st_vol(&S.prio_full, 1);
          ticket = atomicAdd(&P.hdr->dq_head.v, 1u);
          did = true;
        }
      }
    }
    // 2. a static item, when the FIFO has room
    if (!did && room()) {
      if (!main_done) {
        const unsigned q = atomicAdd(&P.hdr->queue.v, 1u);
        if (q >= n_items) {
          main_done = true;
        } else {
          const int rid = __ldg(P.row_list + q / (unsigned)P.nch), chunk = (int)(q % (unsigned)P.nch);
          int kind, b, i;
          decode_row(rid, P.B, P.G, kind, b, i);
          bool take = true;
          if (ld_relaxed(P.known_reject + b) < i) {    // decided reject: the signals may still need the row
            if (!(kind == KIND_DRAFT && P.signals_on)) {
              take = false;
            } else if (defer_on) {                       // to the deferred queue (all CTAs share it)
              const unsigned slot = atomicAdd(&P.hdr->def_tail.v, 1u);
              if (slot < (unsigned)P.def_cap) {
                st_tw(P.defq + slot, tw_make(q, ptag));
                take = false;
              }
            }
          }
          if (take && claim_chunk(P, kind, b, i, chunk, ptag)) push_row(rid, chunk);
          did = true;
        }
      }
      if (!did && main_done && defer_on) {
        if (dticket == 0xffffffffu) dticket = atomicAdd(&P.hdr->def_head.v, 1u);
        if (dticket < (unsigned)P.def_cap) {
          const tword w = ld_tw(P.defq + dticket);
          if (tw_ok(w, ptag)) {
            const unsigned q = tw_u32(w);
            dticket = 0xffffffffu;
            const int rid = __ldg(P.row_list + q / (unsigned)P.nch), chunk = (int)(q % (unsigned)P.nch);
            int kind, b, i;
            decode_row(rid, P.B, P.G, kind, b, i);
            if (claim_chunk(P, kind, b, i, chunk, ptag)) push_row(rid, chunk);
            did = true;
          }
        }
      }
    }
    if (did) {
      idle_since = -1;
      sleep_ns = 32;
      continue;
    }
    // 3. nothing to hand over right now: finished, or dynamic items are
    // still to come (calls without them are finished with the static items)
    if (main_done && (!dyn || ld_relaxed_u32(&P.hdr->done.v) >= n_valid)) break;
    if (ld_relaxed_u32(&P.hdr->error.v) != 0u || aborted(S)) break;
    const long long now = clock64();
    if (idle_since < 0) idle_since = now;
    else if (now - idle_since > P.wait_limit) { ok = false; break; }
    __nanosleep(sleep_ns);
    if (sleep_ns < 256) sleep_ns *= 2;
  }
  if (!ok) {
    set_abort(P, S);
    return;
  }
  // the end marker, once the FIFO has room (bounded)
  const long long c0 = clock64();
  while (!room()) {
    if (aborted(S) || clock64() - c0 > P.wait_limit) {
      set_abort(P, S);
      return;
    }
  }
  push(WT_TERM, 0, 0, 0.f, 0.f);
}

// ---------------------------------------------------------------------------
// consumers

// A direct stage (rows not 16-byte aligned): each consumer thread copies the
// elements of the four vectors it reads itself (load_stage) from global
// memory into the stage buffer, padding past the row's end with -inf.  No
// thread reads another thread's vectors, so no barrier between the consumer
// warps is needed (a warp that gave up on a wait can never leave another
// waiting at one).
template <int DT>
__device__ __forceinline__ void fill_direct(const Params& P, VSmem& S, int stage, const StageDesc& d, int tid) {
  constexpr int N = VecT<DT>::N;
  const ItemDesc& it = S.item[d.item & (kItemSlots - 1)];
  const int kind = (d.item >> 4) & 1;
  const unsigned char* tens = kind == KIND_TARGET ? P.target : P.draft;
  const long long src_elem = row_elem_offset(kind, it.b, it.i, P.G, P.V) + d.elem0;
  const int n = min(stage_elems(DT), P.V - d.elem0);
#pragma unroll 1
  for (int r = 0; r < kVecPerThread; ++r) {
    const int v = tid + r * kConsumerThreads;
    if (v >= d.nvec) break;                   // load_stage pads these itself
#pragma unroll 1
    for (int k = 0; k < N; ++k) {
      const int e = v * N + k;
      if (DT == SPEC_BF16)
        reinterpret_cast<unsigned short*>(S.ring[stage])[e] =
            e < n ? __ldg(reinterpret_cast<const unsigned short*>(tens) + src_elem + e) : (unsigned short)0xff80u;
      else
        reinterpret_cast<float*>(S.ring[stage])[e] =
            e < n ? __ldg(reinterpret_cast<const float*>(tens) + src_elem + e) : -INFINITY;
    }
  }
  __syncwarp();   // orders the element stores before the vector loads that read them back
}

// Residual weight [p - q]_+ of one element pair, p = 2^{x_p c - m_p c} / s_p
// and q likewise: one rounding order everywhere (the scalar form and the
// packed pair form give the same bits), so the slice and group sums and
// the token search agree term by term.
struct ResidW {
  float c, ks, mpc, mqc, rp, nrq;   // nrq = -1 / s_q; ks: see ref_of
  __device__ __forceinline__ float operator()(float xp, float xq) const {
    const float p = ex2(stretch(fmaf(xp, c, -mpc), ks));
    const float q = ex2(stretch(fmaf(xq, c, -mqc), ks));
    return fmaxf(fmaf(p, rp, __fmul_rn(q, nrq)), 0.f);
  }
  __device__ __forceinline__ float2 pair(float2 xp, float2 xq) const {
    const float2 C = make_float2(c, c), K = make_float2(ks, ks);
    float2 a = __ffma2_rn(xp, C, make_float2(-mpc, -mpc));
    float2 b = __ffma2_rn(xq, C, make_float2(-mqc, -mqc));
    a = __ffma2_rn(a, K, a);
    b = __ffma2_rn(b, K, b);
    const float2 p = make_float2(ex2(a.x), ex2(a.y));
    const float2 q = make_float2(ex2(b.x), ex2(b.y));
    const float2 d = __ffma2_rn(p, make_float2(rp, rp), __fmul2_rn(q, make_float2(nrq, nrq)));
    return make_float2(fmaxf(d.x, 0.f), fmaxf(d.y, 0.f));
  }
};

// fp32 weight of a p draw (DK_PF): 2^{stretch(fl(x c - R(m_p)))}, in the
// same rounding order in the scalar and packed forms.
struct PW {
  float c, ks, mpc;
  __device__ __forceinline__ float operator()(float x) const { return ex2(stretch(fmaf(x, c, -mpc), ks)); }
  __device__ __forceinline__ float2 pair(float2 x) const {
    float2 a = __ffma2_rn(x, make_float2(c, c), make_float2(-mpc, -mpc));
    a = __ffma2_rn(a, make_float2(ks, ks), a);
    return make_float2(ex2(a.x), ex2(a.y));
  }
};

// ---------------------------------------------------------------------------
// extended precision for the draw weights
//
// A draw picks the smallest token whose cumulative weight exceeds u W.  A
// vocabulary of V ~ 1.5e5 tokens has as many bucket edges in [0, W), so fp32
// weights (each off by up to half an ulp, 6e-8) move some edge across t in a
// few draws per ten thousand.  Extended-precision weights are computed as an
// unevaluated sum hi + lo of two fp32 values (about 1e-10 relative) and
// summed with error-free transformations, so draws agree with an exact
// (fp64) computation except within ~1e-11 W of an edge.

struct DF {
  float hi, lo;
};

// a + b = s + e exactly (Knuth's two-sum)
__device__ __forceinline__ DF two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  const float bb = __fsub_rn(s, a);
  const float e = __fadd_rn(__fsub_rn(a, __fsub_rn(s, bb)), __fsub_rn(b, bb));
  return {s, e};
}

// a + b = s + e exactly when |a| >= |b| or a = 0
__device__ __forceinline__ DF fast_two_sum(float a, float b) {
  const float s = __fadd_rn(a, b);
  return {s, __fsub_rn(b, __fsub_rn(s, a))};
}

// x + w for non-negative x, w (x normalised, |w.lo| small against w.hi)
__device__ __forceinline__ DF df_add(DF x, DF w) {
  const DF s = two_sum(x.hi, w.hi);
  return fast_two_sum(s.hi, __fadd_rn(s.lo, __fadd_rn(x.lo, w.lo)));
}

// a * b (the product of the high parts exactly, the cross terms rounded once)
__device__ __forceinline__ DF df_mul(DF a, DF b) {
  const float p = __fmul_rn(a.hi, b.hi);
  const float e = __fmaf_rn(a.hi, b.hi, -p);
  return {p, __fmaf_rn(a.hi, b.lo, __fmaf_rn(a.lo, b.hi, e))};
}

// max(p - q, 0), normalised
__device__ __forceinline__ DF df_pos_diff(DF p, DF q) {
  const DF s = two_sum(p.hi, -q.hi);
  const DF d = two_sum(s.hi, __fadd_rn(s.lo, __fsub_rn(p.lo, q.lo)));
  return d.hi > 0.f ? d : DF{0.f, 0.f};
}

__device__ __forceinline__ double df_to_double(DF x) { return (double)x.hi + (double)x.lo; }

// The exponent (x - m) k for a logit x of a row with max m and the scale
// k = k_hi + k_lo = log2(e) / T: x - m by two-sum (not always exact in fp32
// when x is far below m), then a product in extended precision.  -inf for a
// logit of -inf.
__device__ __forceinline__ DF df_exponent(float x, float m, float k_hi, float k_lo) {
  if (!(x > -INFINITY)) return {-INFINITY, 0.f};
  const DF d = two_sum(x, -m);
  const float p = __fmul_rn(d.hi, k_hi);
  const float e = __fmaf_rn(d.hi, k_hi, -p);
  return fast_two_sum(p, __fadd_rn(e, __fmaf_rn(d.hi, k_lo, __fmul_rn(d.lo, k_hi))));
}

// 2^a for a <= 0 given as hi + lo, as hi + lo with about 1e-10 relative error
// (table-driven, after Tang, ACM TOMS 15(2), 1989): a = n + i/256 + r with
// integer n, 0 <= i < 256 and |r| <= 1/512; 2^a = 2^n 2^{i/256} e^{g},
// g = r ln 2, e^g - 1 = g + g^2/2 + g^3/6 (|g| < 0.0014: the next term is
// below 2e-13).  Weights below 2^-126 of the row max are 0.
__device__ __forceinline__ DF exp2_df(DF a, const float2* tab) {
  if (!(a.hi >= -126.f)) return {0.f, 0.f};
  const float j = rintf(__fmul_rn(a.hi, 256.f));
  const int ji = (int)j;
  const int n = ji >> 8, i = ji & 255;                     // ji = 256 n + i, floor division
  // a.hi - j/256 is exact (a multiple of ulp(a.hi), at most 2^-9 in size)
  const float r = __fadd_rn(__fmaf_rn(j, -0.00390625f, a.hi), a.lo);
  const float gh = __fmul_rn(r, kLn2Hi);
  const float gl = __fmaf_rn(r, kLn2Hi, -gh) + __fmul_rn(r, kLn2Lo);  // g = gh + gl
  const float rest = __fmaf_rn(__fmul_rn(gh, gh), __fmaf_rn(gh, 0.16666667f, 0.5f), gl);
  const float2 t = tab[i];
  // T (1 + g + rest) = T_hi + [T_hi g_h + (T_hi rest + T_lo (1 + g_h))]
  const float lo = __fmaf_rn(t.x, gh, __fmaf_rn(t.x, rest, __fmaf_rn(t.y, gh, t.y)));
  const float sc = __int_as_float((n + 127) << 23);          // 2^n, n >= -126
  return {__fmul_rn(t.x, sc), __fmul_rn(lo, sc)};
}

// The extended-precision scales and reciprocal sums of one draw round.
struct DrawX {
  float m1, m2;                     // row maxima (target, draft)
  float k_hi, k_lo;                 // log2(e) / T
  DF r1, r2;                        // 1 / S_p, 1 / S_q (DK_PRESID)
  int excl;                         // token with weight 0 (DK_P), or -1
  int kind;
};

// Extended-precision weight of one token for a DK_P or DK_PRESID round (xd:
// the draft logit, residual only); e: its index in the row.
__device__ __forceinline__ DF draw_weight_x(const DrawX& X, float xt, float xd, int e, const float2* tab) {
  const DF wp = exp2_df(df_exponent(xt, X.m1, X.k_hi, X.k_lo), tab);
  if (X.kind == DK_P) return e == X.excl ? DF{0.f, 0.f} : wp;
  const DF wq = exp2_df(df_exponent(xd, X.m2, X.k_hi, X.k_lo), tab);
  return df_pos_diff(df_mul(wp, X.r1), df_mul(wq, X.r2));
}

// Warp-wide extended-precision sum (xor butterfly; every lane ends with it)
__device__ __forceinline__ DF warp_sum_df(DF v) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    DF o;
    o.hi = __shfl_xor_sync(0xffffffffu, v.hi, off);
    o.lo = __shfl_xor_sync(0xffffffffu, v.lo, off);
    v = df_add(v, o);
  }
  return v;
}

// Four sums over the warp's 32 lanes in six shuffles (the values are halved
// across lanes at the first two steps): lane l ends with the total of
// v[(l >> 3) & 3].
__device__ __forceinline__ float warp_sum4(const float (&v)[4], int lane) {
  const bool h16 = (lane & 16) != 0, h8 = (lane & 8) != 0;
  const float k0 = (h16 ? v[2] : v[0]) + __shfl_xor_sync(0xffffffffu, h16 ? v[0] : v[2], 16);
  const float k1 = (h16 ? v[3] : v[1]) + __shfl_xor_sync(0xffffffffu, h16 ? v[1] : v[3], 16);
  float k = (h8 ? k1 : k0) + __shfl_xor_sync(0xffffffffu, h8 ? k0 : k1, 8);
  k += __shfl_xor_sync(0xffffffffu, k, 4);
  k += __shfl_xor_sync(0xffffffffu, k, 2);
  k += __shfl_xor_sync(0xffffffffu, k, 1);
  return k;
}

// One slice of an extended-precision draw round (DK_P, DK_SUMS, DK_PRESID)
// by the 8 consumer warps (warp-wide).  DK_P / DK_PRESID: each group's sum
// (fp64, two tagged words) and, in *ds1, this warp's part of the slice sum.
// DK_SUMS: this warp's parts of S_p (*ds1) and S_q (*ds2).  Vectors past
// the row read as -inf and weigh 0.
template <int DT>
__device__ __forceinline__ void draw_slice_x(const Params& P, const ItemDesc& it, const float2* tab, const uint4* vec,
                                             const uint4* vec2, int elem0, int nvec, int cw, int lane, double* ds1,
                                             double* ds2) {
  constexpr int N = VecT<DT>::N;
  const int tid = cw * 32 + lane;
  DrawX X;
  X.m1 = it.m1; X.m2 = it.m2; X.k_hi = it.c; X.k_lo = it.c_lo;
  X.r1 = DF{it.r1h, it.r1l}; X.r2 = DF{it.r2h, it.r2l};
  X.excl = it.y; X.kind = it.aux;
  const bool two = X.kind != DK_P;
  tword* gs_out = P.gsum + ((size_t)it.b * P.nres + it.chunk) * kGroupsPerStage * kGroupWords;
  DF sp{0.f, 0.f}, sq{0.f, 0.f};
  double s = 0.0;
  // one vector (and group) at a time: the extended arithmetic keeps few
  // registers live
#pragma unroll 1
  for (int q = 0; q < kVecPerThread; ++q) {
    const int v = tid + q * kConsumerThreads;
    const uint4 pad = DT == SPEC_BF16 ? make_uint4(0xff80ff80u, 0xff80ff80u, 0xff80ff80u, 0xff80ff80u)
                                      : make_uint4(0xff800000u, 0xff800000u, 0xff800000u, 0xff800000u);
    float xt[N], xd[N];
    VecT<DT>::unpack(v < nvec ? vec[v] : pad, xt);
    if (two) VecT<DT>::unpack(v < nvec ? vec2[v] : pad, xd);
    // (rare rounds: the loops over a vector's tokens are not unrolled, which
    // keeps their code out of the way of the streaming loop)
    if (X.kind == DK_SUMS) {
#pragma unroll 1
      for (int k = 0; k < N; ++k) {
        sp = df_add(sp, exp2_df(df_exponent(xt[k], X.m1, X.k_hi, X.k_lo), tab));
        sq = df_add(sq, exp2_df(df_exponent(xd[k], X.m2, X.k_hi, X.k_lo), tab));
      }
      continue;
    }
    DF acc{0.f, 0.f};
#pragma unroll 1
    for (int k = 0; k < N; ++k)
      acc = df_add(acc, draw_weight_x(X, xt[k], two ? xd[k] : 0.f, elem0 + v * N + k, tab));
    // group cw + 8 q (the vectors 32 cw + 256 q + lane): lane 0 publishes it
    const DF g = warp_sum_df(acc);
    if ((cw + 8 * q) * kGroupVecs < nvec) {
      const double gv = df_to_double(g);
      s += gv;
      if (lane == 0) {
        const unsigned long long bits = (unsigned long long)__double_as_longlong(gv);
        tword* o = gs_out + (cw + 8 * q) * kGroupWords;
        st_tw(o, tw_make((unsigned)(bits >> 32), it.tag));
        st_tw(o + 1, tw_make((unsigned)bits, it.tag));
      }
    }
  }
  if (X.kind == DK_SUMS) {
    *ds1 = df_to_double(warp_sum_df(sp));
    *ds2 = df_to_double(warp_sum_df(sq));
  } else {
    *ds1 = s;
    *ds2 = 0.0;
  }
}

struct SliceSums {
  double s1, s2;
};

template <int DT>
__device__ __forceinline__ SliceSums draw_slice(const Params& P, const ItemDesc& it, const uint4* vec, const uint4* vec2,
                                                int elem0, int nvec, int cw, int lane) {
  SliceSums out{0.0, 0.0};
  if (it.aux != DK_RESID && it.aux != DK_PF) {
    extern __shared__ __align__(128) unsigned char smem_raw[];
    const float2* tab = reinterpret_cast<const VSmem*>(smem_raw)->exp2tab;
    draw_slice_x<DT>(P, it, tab, vec, vec2, elem0, nvec, cw, lane, &out.s1, &out.s2);
    return out;
  }
  constexpr int N = VecT<DT>::N;
  const int tid = cw * 32 + lane;
  const unsigned dtag = it.tag;
  const StageDesc d{0, nvec, elem0, 0};
  double dsum = 0.0;
  const bool pf = it.aux == DK_PF;
  uint4 wt[kVecPerThread], wd[kVecPerThread];
  load_stage<DT>(vec, d.nvec, tid, wt);
  if (!pf) load_stage<DT>(vec2, d.nvec, tid, wd);
  ResidW R;
  R.c = it.c; R.ks = scale_k(it.c, it.c_lo); R.mpc = ref_of(it.m1, it.c); R.mqc = ref_of(it.m2, it.c);
  R.rp = 1.f / it.s1; R.nrq = -1.f / it.s2;
  const PW Wp{R.c, R.ks, R.mpc};
  const int excl = it.y;            // DK_PF: the token left out (one-hot residual), or -1
  tword* gs_out = P.gsum + ((size_t)it.b * P.nres + it.chunk) * kGroupsPerStage * kGroupWords;
  float gq[kVecPerThread];          // the lane's vector sums
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) {
    float xt[N], xd[N], e[N];
    VecT<DT>::unpack(wt[q], xt);
    if (pf) {
      const int base = elem0 + (tid + q * kConsumerThreads) * N;
#pragma unroll
      for (int k = 0; k < N; k += 2) {
        const float2 w2 = Wp.pair(make_float2(xt[k], xt[k + 1]));
        e[k] = base + k == excl ? 0.f : w2.x;
        e[k + 1] = base + k + 1 == excl ? 0.f : w2.y;
      }
    } else {
      VecT<DT>::unpack(wd[q], xd);
#pragma unroll
      for (int k = 0; k < N; k += 2) {
        const float2 w2 = R.pair(make_float2(xt[k], xt[k + 1]), make_float2(xd[k], xd[k + 1]));
        e[k] = w2.x; e[k + 1] = w2.y;
      }
    }
    if (N == 8) gq[q] = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
    else gq[q] = (e[0] + e[1]) + (e[2] + e[3]);
  }
  // the vectors 32 cw + 256 q + lane of one warp form group cw + 8 q; lane
  // 8 q ends with its sum and publishes it (as an fp64, two words)
  const float gsum = warp_sum4(gq, lane);
  if ((lane & 7) == 0 && (cw + (lane >> 3) * 8) * kGroupVecs < d.nvec) {
    const unsigned long long bits = (unsigned long long)__double_as_longlong((double)gsum);
    tword* o = gs_out + (cw + (lane >> 3) * 8) * kGroupWords;
    st_tw(o, tw_make((unsigned)(bits >> 32), dtag));
    st_tw(o + 1, tw_make((unsigned)bits, dtag));
  }
  const float g1 = __shfl_sync(0xffffffffu, gsum, 8), g2 = __shfl_sync(0xffffffffu, gsum, 16),
              g3 = __shfl_sync(0xffffffffu, gsum, 24);
  const float gg[kVecPerThread] = {gsum, g1, g2, g3};
  if (lane == 0)
#pragma unroll
    for (int q = 0; q < kVecPerThread; ++q)
      if ((cw + 8 * q) * kGroupVecs < d.nvec) dsum += (double)gg[q];
  out.s1 = dsum;
  return out;
}

template <int DT, bool GREEDY>
__device__ __forceinline__ void consumer_role(const Params& P, VSmem& S, int cw, int lane) {
  constexpr int N = VecT<DT>::N;
  const int tid = cw * 32 + lane;
  int stage = 0;
  uint32_t phase = 0;
  int seq = 0;
  RunState r;
  run_reset(r);
  auto advance = [&]() {
    if (++stage == kStages) { stage = 0; phase ^= 1u; }
  };
  auto release = [&](int st) {
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[st]);
  };
  // hand one finished item to the epilogue warps
  auto to_epilogue = [&](auto write_fields) -> bool {
    const int eslot = seq % kEpiSlots;
    const uint32_t round = (uint32_t)(seq / kEpiSlots) & 1u;
    if (!wait_bar(S, &S.epi_empty[eslot], round ^ 1u)) { set_abort(P, S); return false; }
    write_fields(S.slot[eslot]);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.epi_full[eslot]);
    ++seq;
    return true;
  };
  while (true) {
    if (!wait_bar(S, &S.full[stage], phase)) { set_abort(P, S); return; }
    const StageDesc d = S.desc[stage];
    if (d.flags & F_TERM) {
      // every epilogue warp must see the end: mark consecutive slots
      for (int e = 0; e < kEpiWarps; ++e) {
        if (!to_epilogue([&](EpiSlot& E) { if (tid == 0) E.term = 1; })) return;
      }
      return;
    }
    if (d.flags & F_DIRECT) fill_direct<DT>(P, S, stage, d, tid);
    const uint4* vec = reinterpret_cast<const uint4*>(S.ring[stage]);

    if (!(d.flags & F_DRAW)) {
      const ItemDesc& it = S.item[d.item & (kItemSlots - 1)];
      if (d.flags & F_FIRST) run_reset(r);
      // the item's scale and entropy flag are read from shared memory at
      // every stage (no consumer register holds them across stages)
      const bool ent = !GREEDY && it.kind == KIND_DRAFT && P.signals_on;
      const float c = it.c, ks = it.ks;
      uint4 w[kVecPerThread];
      load_stage<DT>(vec, d.nvec, tid, w);
      if (GREEDY) stage_argmax<DT>(r, w, d.elem0, tid);
      else if (ent) stage_softmax<DT, true>(r, w, c, ks);
      else stage_softmax<DT, false>(r, w, c, ks);
      release(stage);
      advance();
      if (d.flags & F_LAST) {
        if (tid == 0 && (it.nhead > 0 || it.ntail > 0)) {
          const unsigned char* tens = it.kind == KIND_TARGET ? P.target : P.draft;
          const long long row0 = row_elem_offset(it.kind, it.b, it.i, P.G, P.V);
          for (int k = 0; k < it.nhead; ++k) {
            run_scalar<GREEDY>(r, load_logit(tens, DT, row0 + it.head0 + k), it.head0 + k, c, ks, ent);
          }
          for (int k = 0; k < it.ntail; ++k) {
            run_scalar<GREEDY>(r, load_logit(tens, DT, row0 + it.tail0 + k), it.tail0 + k, c, ks, ent);
          }
        }
        Part p;
        if (GREEDY) {
          p = to_part(r);
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) p = merge_argmax(p, shfl_part(p, off));
        } else {
          p = warp_softmax_part(r, c, ks, ent);
        }
        if (!to_epilogue([&](EpiSlot& E) {
              if (lane == 0) E.part[cw] = p;
              if (tid == 0) {
                E.type = IT_STATS; E.row_id = it.row_id; E.b = it.b; E.i = it.i; E.kind = it.kind;
                E.chunk = it.chunk; E.c = c; E.ks = ks;
              }
            }))
          return;
      }
      continue;
    }

    // IT_DSUM: one slice of a draw round (a stage pair when it reads rows k
    // of both models); greedy calls have no draws
    if constexpr (GREEDY) continue;
    const ItemDesc& it = S.item[d.item & (kItemSlots - 1)];
    const int dk = it.aux;
    const bool two = dk != DK_P && dk != DK_PF;
    const int st1 = stage;
    const uint4* vec2 = vec;
    if (two) {
      advance();
      if (!wait_bar(S, &S.full[stage], phase)) { set_abort(P, S); return; }
      const StageDesc d2 = S.desc[stage];
      if (d2.flags & F_DIRECT) fill_direct<DT>(P, S, stage, d2, tid);
      vec2 = reinterpret_cast<const uint4*>(S.ring[stage]);
    }
    const unsigned dtag = it.tag;
    // lane 0: this warp's part of the slice sum(s)
    const SliceSums ds = draw_slice<DT>(P, it, vec, vec2, d.elem0, d.nvec, cw, lane);
    release(st1);
    if (two) release(stage);
    advance();
    if (!to_epilogue([&](EpiSlot& E) {
          if (lane == 0) { E.dsum[cw] = ds.s1; E.dsum2[cw] = ds.s2; }
          if (tid == 0) { E.type = IT_DSUM; E.b = it.b; E.chunk = it.chunk; E.i = it.i; E.kind = dk; E.tag = dtag; }
        }))
      return;
  }
}

// ---------------------------------------------------------------------------
// epilogue: publish chunk partials and draw slice sums as tagged words

template <int DT, bool GREEDY>
__device__ __forceinline__ void epilogue_role(const Params& P, VSmem& S, int lane, int e, unsigned epoch) {
  const int nch = P.nch;
  for (int seq = e;; seq += kEpiWarps) {
    const int eslot = seq % kEpiSlots;
    const uint32_t epar = (uint32_t)(seq / kEpiSlots) & 1u;
    if (!wait_bar(S, &S.epi_full[eslot], epar)) { set_abort(P, S); return; }
    const EpiSlot& E = S.slot[eslot];
    if (E.term) return;
    const int type = E.type, rid = E.row_id, b = E.b, kind = E.kind, chunk = E.chunk;
    const float c = E.c, ks = E.ks;
    const unsigned dtag = E.tag;
    Part p = lane < kConsumerWarps ? E.part[lane] : empty_part();
    double ws = 0.0, ws2 = 0.0;
    if (lane == 0 && type == IT_DSUM)
      for (int w = 0; w < kConsumerWarps; ++w) { ws += E.dsum[w]; ws2 += E.dsum2[w]; }
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.epi_empty[eslot]);

    if (type == IT_DSUM) {
      // the slice sum (DK_SUMS: S_p and S_q parts), fp64 as two tagged halves each
      if (lane == 0) {
        tword* o = P.dsum + kSliceWords * ((size_t)b * P.nres + chunk);
        unsigned long long bits = (unsigned long long)__double_as_longlong(ws);
        st_tw(o, tw_make((unsigned)(bits >> 32), dtag));
        st_tw(o + 1, tw_make((unsigned)bits, dtag));
        if (kind == DK_SUMS) {
          bits = (unsigned long long)__double_as_longlong(ws2);
          st_tw(o + 2, tw_make((unsigned)(bits >> 32), dtag));
          st_tw(o + 3, tw_make((unsigned)bits, dtag));
        }
      }
      continue;
    }
    // IT_STATS: merge the consumer warps' partials (lanes 0..7), publish.
    // Softmax partials: the max first, one rescale of each partial to it,
    // then plain sums (fixed xor tree: deterministic).
    if (GREEDY) {
#pragma unroll
      for (int off = 4; off >= 1; off >>= 1) p = merge_argmax(p, shfl_part(p, off));
    } else {
      const bool ent = kind == KIND_DRAFT && P.signals_on;
      float m = p.m;
#pragma unroll
      for (int off = 4; off >= 1; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
      float ss = 0.f, tt = 0.f;
      if (p.s != 0.f) {            // an empty partial contributes 0
        const float dd = stretch(__fsub_rn(ref_of(p.m, c), ref_of(m, c)), ks);
        const float f = ex2(dd);
        ss = p.s * f;
        if (ent) tt = f * fmaf(dd, p.s, p.t);
      }
#pragma unroll
      for (int off = 4; off >= 1; off >>= 1) {
        ss += __shfl_xor_sync(0xffffffffu, ss, off);
        if (ent) tt += __shfl_xor_sync(0xffffffffu, tt, off);
      }
      p.m = m; p.s = ss; p.t = tt;
    }
    if (lane == 0) {
      tword* o = P.cparts + ((size_t)rid * nch + chunk) * kPartWords;
      const unsigned ptag = part_tag(epoch);
      st_tw(o + 0, tw_make(__float_as_uint(p.m), ptag));
      st_tw(o + 1, tw_make(GREEDY ? (unsigned)p.idx : __float_as_uint(p.s), ptag));
      if (!GREEDY) st_tw(o + 2, tw_make(__float_as_uint(p.t), ptag));
    }
  }
}

// ---------------------------------------------------------------------------
// owner: one warp per CTA takes each of its requests (b = CTA, CTA + grid,
// ...) from the row partials to the outputs: merges the rows in the order
// the schedule streams them, tests the positions in order, publishes the
// first reject (early exit), runs the draw and writes the outputs.  All of a
// request's decisions are taken in one warp, so they need no atomics.

// A wait of the owner gives up after P.wait_limit cycles, or at once when any
// role of any CTA has given up (the header error word).
struct OwnerClock {
  long long c0;
  int polls;
  __device__ __forceinline__ void start() { c0 = clock64(); polls = 0; }
  __device__ __forceinline__ bool expired(const Params& P) {
    const bool mine = __any_sync(0xffffffffu, clock64() - c0 > P.wait_limit);
    if (mine) {   // this wait gave up: every other role gives up too
      if ((threadIdx.x & 31) == 0) atomicOr(&P.hdr->error.v, (unsigned)SPEC_ST_TIMEOUT);
      return true;
    }
    // the error word of the other roles is read every 8th poll only (a read
    // per poll would double the round trips of every poll)
    if ((++polls & 7) != 0) return false;
    return __any_sync(0xffffffffu, ld_relaxed_u32(&P.hdr->error.v) != 0u);
  }
};

struct RowRes {
  RowStats st;   // merged statistics (every lane)
  float xy;      // logit at the draft token (NaN if not loaded)
};

// Tagged words of a chunk partial that carry data, and the partial they hold.
template <bool GREEDY>
__host__ __device__ constexpr int part_words() { return GREEDY ? 2 : 3; }
template <bool GREEDY>
__device__ __forceinline__ Part part_of(const tword (&w)[kPartWords]) {
  Part q;
  q.m = tw_f32(w[0]);
  if (GREEDY) {
    q.idx = (int)tw_u32(w[1]);
    q.s = q.t = 0.f;
  } else {
    q.s = tw_f32(w[1]);
    q.t = tw_f32(w[2]);
    q.idx = 0x3fffffff;
  }
  return q;
}

// Merged statistics of row rid (warp-wide).  Waits until every chunk
// partial carries the call's tag and merges them in chunk order (lane l
// takes chunks l, l+32, ...; then a fixed xor tree).  False if the wait gave
// up.
template <bool GREEDY>
__device__ bool merge_row(const Params& P, int rid, float c, float ks, bool ent, unsigned epoch, int lane, RowRes& out) {
  constexpr int NW = part_words<GREEDY>();
  const int nch = P.nch;
  const tword* base = P.cparts + (size_t)rid * nch * kPartWords;
  Part r = empty_part();
  OwnerClock clk;
  clk.start();
  for (int k0 = 0; k0 < nch; k0 += 32) {
    const int k = k0 + lane;
    tword w[kPartWords] = {};
    while (true) {
      bool ok = true;
      if (k < nch) {
#pragma unroll
        for (int j = 0; j < NW; ++j) {
          w[j] = ld_tw(base + (size_t)k * kPartWords + j);
          ok &= tw_ok(w[j], part_tag(epoch));
        }
      }
      if (__all_sync(0xffffffffu, ok)) break;
      if (clk.expired(P)) return false;
    }
    if (k < nch) r = GREEDY ? merge_argmax(r, part_of<GREEDY>(w)) : merge_parts(r, part_of<GREEDY>(w), c, ks, ent);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) {
    const Part o = shfl_part(r, off);
    r = GREEDY ? merge_argmax(r, o) : merge_parts(r, o, c, ks, ent);
  }
  out.st.m = r.m; out.st.s = r.s; out.st.t = r.t; out.st.idx = r.idx;
  out.xy = qnan();
  return true;
}

// Target row ridT and draft row ridD of one position, merged together
// (warp-wide; needs 2 * nch <= 32): lanes 0-15 take the target's chunks,
// lanes 16-31 the draft's, so one poll covers both rows.  Each half merges
// with the same tree as merge_row (its xor-16 level only meets empty
// partials, which merge exactly), so the results are identical to two
// merge_row calls.  False if the wait gave up.
__device__ bool merge_pair(const Params& P, int ridT, int ridD, float c, float ks, bool entD, unsigned epoch, int lane,
                           RowRes& T, RowRes& D) {
  const int nch = P.nch;
  const int half = lane >> 4, k = lane & 15;
  const tword* base = P.cparts + (size_t)(half ? ridD : ridT) * nch * kPartWords;
  const bool ent = half ? entD : false;
  tword w[kPartWords] = {};
  OwnerClock clk;
  clk.start();
  while (true) {
    bool ok = true;
    if (k < nch) {
#pragma unroll
      for (int j = 0; j < part_words<false>(); ++j) {
        w[j] = ld_tw(base + (size_t)k * kPartWords + j);
        ok &= tw_ok(w[j], part_tag(epoch));
      }
    }
    if (__all_sync(0xffffffffu, ok)) break;
    if (clk.expired(P)) return false;
  }
  Part r = empty_part();
  if (k < nch) r = merge_parts(r, part_of<false>(w), c, ks, ent);
#pragma unroll
  for (int off = 8; off >= 1; off >>= 1) r = merge_parts(r, shfl_part(r, off), c, ks, ent);
  T.st.m = __shfl_sync(0xffffffffu, r.m, 0);  T.st.s = __shfl_sync(0xffffffffu, r.s, 0);
  T.st.t = __shfl_sync(0xffffffffu, r.t, 0);  T.st.idx = __shfl_sync(0xffffffffu, r.idx, 0);
  D.st.m = __shfl_sync(0xffffffffu, r.m, 16); D.st.s = __shfl_sync(0xffffffffu, r.s, 16);
  D.st.t = __shfl_sync(0xffffffffu, r.t, 16); D.st.idx = __shfl_sync(0xffffffffu, r.idx, 16);
  T.xy = D.xy = qnan();
  return true;
}

// Up to four rows at once (warp-wide; needs nch <= 8): row s in lanes
// 8s .. 8s+7, given per lane by its segment's row id (< 0: no row) and
// entropy flag.  Segments in need_mask are waited for; the others are taken
// only if already complete.  Each row merges with the same tree as
// merge_row (its xor-16 and xor-8 levels only meet empty partials, which
// merge exactly), so results are identical.  Every lane of segment s ends
// with row s's statistics in pm.  Returns the mask of the segments taken
// (absent rows count as taken), or -1 if the wait gave up.
template <bool GREEDY>
__device__ int merge_rows4(const Params& P, int rid, bool ent, unsigned need_mask, float c, float ks, unsigned epoch,
                           int lane, Part& pm) {
  constexpr int NW = part_words<GREEDY>();
  const int nch = P.nch;
  const int seg = lane >> 3, k = lane & 7;
  const bool has = rid >= 0 && k < nch;
  const tword* base = P.cparts + ((size_t)(rid < 0 ? 0 : rid) * nch + k) * kPartWords;
  tword w[kPartWords] = {};
  unsigned ready = 0;
  OwnerClock clk;
  clk.start();
  while (true) {
    bool ok = true;
    if (has) {
#pragma unroll
      for (int j = 0; j < NW; ++j) {
        w[j] = ld_tw(base + j);
        ok &= tw_ok(w[j], part_tag(epoch));
      }
    }
    const unsigned bal = __ballot_sync(0xffffffffu, ok);
    ready = 0;
#pragma unroll
    for (int s2 = 0; s2 < 4; ++s2)
      if (((bal >> (8 * s2)) & 0xffu) == 0xffu) ready |= 1u << s2;
    if ((ready & need_mask) == need_mask) break;
    if (clk.expired(P)) return -1;
  }
  const bool take = has && ((ready >> seg) & 1u);
  Part r = empty_part();
  if (take) r = GREEDY ? merge_argmax(r, part_of<GREEDY>(w)) : merge_parts(r, part_of<GREEDY>(w), c, ks, ent);
#pragma unroll
  for (int off = 4; off >= 1; off >>= 1) {
    const Part o = shfl_part(r, off);
    r = GREEDY ? merge_argmax(r, o) : merge_parts(r, o, c, ks, ent);
  }
  pm = r;
  return (int)ready;
}

// Row s of a merge_rows4 result, as every lane sees it (x_y not loaded).
__device__ __forceinline__ RowRes row_of(const Part& pm, int s) {
  RowRes o;
  o.st.m = __shfl_sync(0xffffffffu, pm.m, 8 * s);
  o.st.s = __shfl_sync(0xffffffffu, pm.s, 8 * s);
  o.st.t = __shfl_sync(0xffffffffu, pm.t, 8 * s);
  o.st.idx = __shfl_sync(0xffffffffu, pm.idx, 8 * s);
  o.xy = qnan();
  return o;
}

__device__ __forceinline__ int status_of_code(int code) {
  return code == PC_NONFINITE ? SPEC_ST_NONFINITE
       : code == PC_BAD_TOKEN ? SPEC_ST_BAD_TOKEN
       : code == PC_BAD_UNIFORM ? SPEC_ST_BAD_UNIFORM : SPEC_ST_TIMEOUT;
}

// Acceptance test of position i (tutorial page "5.1 投机解码核心原理",
// sections 3.1-3.3), in fp32 on the merged row statistics:
//   p(y) = 2^{a(x_y)} / s_p with the exponent a of every term of s_p (see
//   ref_of), q(y) likewise (1 for one-hot q),
//   accept <=> u q(y) < p(y),  a = min(1, p(y)/q(y)).
// A test closer than 1e-5 (relative) to its threshold is counted; it is not
// published as an early exit.  Returns the position code (with
// PC_UNCERTAIN); *a = a_i (NaN when not computed).  Every lane computes the
// same.
template <bool GREEDY>
__device__ int evaluate_pos(const Params& P, int b, int i, const RowRes& T, const RowRes& D, int y, float c,
                            float ks, float* a_out) {
  const int G = P.G, V = P.V;
  int code;
  float a = qnan();
  if (GREEDY) {
    if (!row_ok(T.st, true)) code = PC_NONFINITE;
    else if (y < 0 || y >= V) code = PC_BAD_TOKEN;
    else code = (y == (T.st.idx & ~kIdxNaN)) ? PC_ACCEPT : PC_REJECT;
  } else {
    const bool sample = P.mode == MODE_SAMPLE;
    const float u = P.uniforms[(size_t)b * (G + 1) + i];
    if (!row_ok(T.st, false) || (sample && !row_ok(D.st, false))) code = PC_NONFINITE;
    else if (y < 0 || y >= V) code = PC_BAD_TOKEN;
    else if (!(u >= 0.f && u < 1.f)) code = PC_BAD_UNIFORM;
    else {
      const float py = ex2(stretch(fmaf(T.xy, c, -ref_of(T.st.m, c)), ks)) / T.st.s;
      const float qy = sample ? ex2(stretch(fmaf(D.xy, c, -ref_of(D.st.m, c)), ks)) / D.st.s : 1.f;
      const float uq = u * qy;
      code = uq < py ? PC_ACCEPT : PC_REJECT;
      a = qy > 0.f ? fminf(1.f, py / qy) : (py > 0.f ? 1.f : 0.f);
      if (fabsf(uq - py) <= 1e-5f * fmaxf(uq, py)) code |= PC_UNCERTAIN;
    }
  }
  *a_out = a;
  return code;
}

// Warp-wide: among n non-negative weights get(0..n-1) in order, the first j
// whose prefix (fp64, fixed association) plus weight exceeds t, with the
// prefix before it; when none does, the last j of positive weight (-1 if
// none).  *total = the sum of all weights.
template <class Get>
__device__ int warp_locate(int n, Get get, double t, double* before, double* total, int lane) {
  double carry = 0.0, fb = 0.0, lb = 0.0;
  int found = -1, lastpos = -1;
  for (int base = 0; base < n; base += 32) {
    const int j = base + lane;
    const double v = j < n ? get(j) : 0.0;
    double incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const double o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    double ex = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) ex = 0.0;
    ex += carry;
    const unsigned cross = __ballot_sync(0xffffffffu, j < n && ex + v > t);
    const unsigned pos = __ballot_sync(0xffffffffu, j < n && v > 0.0);
    if (found < 0 && cross) {
      const int f = __ffs(cross) - 1;
      found = base + f;
      fb = __shfl_sync(0xffffffffu, ex, f);
    }
    if (pos) {
      const int l = 31 - __clz(pos);
      lastpos = base + l;
      lb = __shfl_sync(0xffffffffu, ex, l);
    }
    carry += __shfl_sync(0xffffffffu, incl, 31);
  }
  *total = carry;
  if (found >= 0) { *before = fb; return found; }
  *before = lb;
  return lastpos;
}

// Warp inclusive scan of one fp64 value per lane (fixed association).
__device__ __forceinline__ double warp_incl_scan(double v, int lane) {
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const double o = __shfl_up_sync(0xffffffffu, v, d);
    if (lane >= d) v += o;
  }
  return v;
}

// Start one round of the draw of request b: its descriptor (read by the
// producers that stage the slices), then one queue entry per slice of row k.
// Warp-wide.
__device__ void start_draw(const Params& P, int b, int k, const DrawX& X, const RowStats& tr, const RowStats& dr,
                           float c, int round, unsigned epoch, int lane) {
  const unsigned tag = draw_tag(epoch, round);
  tword* dd = P.dd + (size_t)b * kDrawWords;
  unsigned v = 0u;
  if (lane == DW_KIND) v = (unsigned)X.kind | ((unsigned)k << 8);
  else if (lane == DW_EXCL) v = (unsigned)X.excl;
  else if (lane == DW_M1) v = __float_as_uint(tr.m);
  else if (lane == DW_S1) v = __float_as_uint(tr.s);
  else if (lane == DW_M2) v = __float_as_uint(dr.m);
  else if (lane == DW_S2) v = __float_as_uint(dr.s);
  else if (lane == DW_C) v = __float_as_uint(c);
  else if (lane == DW_CLO) v = __float_as_uint(X.k_lo);
  else if (lane == DW_R1H) v = __float_as_uint(X.r1.hi);
  else if (lane == DW_R1L) v = __float_as_uint(X.r1.lo);
  else if (lane == DW_R2H) v = __float_as_uint(X.r2.hi);
  else if (lane == DW_R2L) v = __float_as_uint(X.r2.lo);
  if (lane < DW_END) st_tw(dd + lane, tw_make(v, tag));
  __syncwarp();
  enqueue_draw(P, P.nres, b, round, epoch, lane);
}

enum DrawResult : int { DR_OK = 0, DR_ZERO = 1, DR_FAIL = 2 };

__device__ __forceinline__ double word_pair_f64(tword a, tword b) {
  return __longlong_as_double((long long)(((unsigned long long)tw_u32(a) << 32) | tw_u32(b)));
}

// The fp64 at words j, j+1 of an array of tagged words
__device__ __forceinline__ double tagged_f64(const tword* o, int j) { return word_pair_f64(ld_tw(o + j), ld_tw(o + j + 1)); }

// Waits until the first `words` tagged words of every slice sum of request
// b's round carry `tag` (warp-wide); false if the wait gave up.
__device__ bool wait_slices(const Params& P, int b, unsigned tag, int words, int lane) {
  const tword* sums = P.dsum + (size_t)kSliceWords * b * P.nres;
  OwnerClock clk;
  clk.start();
  for (int j0 = 0; j0 < P.nres; j0 += 32) {
    const int j = j0 + lane;
    while (true) {
      bool ok = true;
      if (j < P.nres)
        for (int w = 0; w < words; ++w) ok &= tw_ok(ld_tw(sums + (size_t)kSliceWords * j + w), tag);
      if (__all_sync(0xffffffffu, ok)) break;
      if (clk.expired(P)) return false;
    }
  }
  return true;
}

// The slice and group of a draw round once its slices are summed
// (warp-wide): W = sum of the slice sums (fp64, slice order), t = u W; the
// slice by the fp64 prefix of the slice sums, then the group of 32 vectors
// (256 bf16 / 128 fp32 tokens) by the fp64 prefix of its stored group sums.
struct DrawLoc {
  int r;                            // DR_OK, DR_ZERO (W = 0) or DR_FAIL
  double W, t;
  int e0, g0;                       // first token of the slice and of the group
  double tl2;                       // t less everything before the group
};

template <int DT>
__device__ DrawLoc locate_draw(const Params& P, int b, float ud, unsigned tag, int lane) {
  constexpr int GE = kGroupVecs * VecT<DT>::N;       // tokens per group
  DrawLoc L{};
  L.r = DR_FAIL;
  const int V = P.V, nres = P.nres, se = stage_elems(DT);
  const tword* sums = P.dsum + (size_t)kSliceWords * b * nres;
  if (!wait_slices(P, b, tag, 2, lane)) return L;
  double W, before;
  int cs;
  if (nres <= 32) {
    const double v = lane < nres ? tagged_f64(sums, kSliceWords * lane) : 0.0;
    const double incl = warp_incl_scan(v, lane);
    W = __shfl_sync(0xffffffffu, incl, 31);
    const double t = (double)ud * W;
    const unsigned cross = __ballot_sync(0xffffffffu, lane < nres && incl > t);
    const unsigned pos = __ballot_sync(0xffffffffu, v > 0.0);
    cs = cross ? __ffs(cross) - 1 : (pos ? 31 - __clz(pos) : -1);
    before = cs >= 0 ? __shfl_sync(0xffffffffu, incl - v, cs) : 0.0;
  } else {
    auto get = [&](int j) -> double { return tagged_f64(sums, kSliceWords * j); };
    warp_locate(nres, get, INFINITY, &before, &W, lane);
    double tot;
    cs = warp_locate(nres, get, (double)ud * W, &before, &tot, lane);
  }
  if (!(W > 0.0)) { L.r = DR_ZERO; return L; }
  if (cs < 0) return L;
  const double t = (double)ud * W;
  const int e0 = cs * se, e1 = min(e0 + se, V);
  const int ngroups = (e1 - e0 + GE - 1) / GE;       // <= kGroupsPerStage = 32
  // lane l holds group l of the slice (fp64, two words)
  const tword* gsum = P.gsum + ((size_t)b * nres + cs) * kGroupsPerStage * kGroupWords;
  double gv = 0.0;
  OwnerClock clk;
  clk.start();
  while (true) {
    bool ok = true;
    if (lane < ngroups) {
      const tword w0 = ld_tw(gsum + kGroupWords * lane), w1 = ld_tw(gsum + kGroupWords * lane + 1);
      ok = tw_ok(w0, tag) && tw_ok(w1, tag);
      gv = word_pair_f64(w0, w1);
    }
    if (__all_sync(0xffffffffu, ok)) break;
    if (clk.expired(P)) return L;
  }
  const double lsum = lane < ngroups ? gv : 0.0;
  const double tl = t - before;
  const double gincl = warp_incl_scan(lsum, lane);
  const unsigned gcross = __ballot_sync(0xffffffffu, gincl > tl);
  const unsigned gpos = __ballot_sync(0xffffffffu, lsum > 0.0);
  const int g = gcross ? __ffs(gcross) - 1 : (gpos ? 31 - __clz(gpos) : 0);
  L.tl2 = tl - __shfl_sync(0xffffffffu, gincl - lsum, g);
  L.W = W;
  L.t = t;
  L.e0 = e0;
  L.g0 = e0 + g * GE;
  L.r = DR_OK;
  return L;
}

// The token inside the located group from its recomputed weights w[0..PER)
// per lane (lane l: tokens g0 + l PER ...): the first whose fp64 prefix
// exceeds tl2, with the distance of tl2 from the nearer edge of its bucket;
// if rounding leaves no crossing, the group's last token of positive weight
// (margin 0).  Warp-wide; z = -1 if the group has no weight at all.
template <int PER>
__device__ int walk_group(const double (&w)[PER], int g0, double tl2, double* margin_out, int lane) {
  double mine = 0.0;
#pragma unroll
  for (int u = 0; u < PER; ++u) mine += w[u];
  const double incl = warp_incl_scan(mine, lane);
  const double ex = incl - mine;
  const unsigned cross = __ballot_sync(0xffffffffu, incl > tl2);
  int z = -1;
  double margin = 0.0;
  if (cross) {
    const int f = __ffs(cross) - 1;
    if (lane == f) {
      double C = ex, Cp = ex;
      for (int u = 0; u < PER; ++u) {
        Cp = C;
        C += w[u];
        if (C > tl2) { z = g0 + lane * PER + u; break; }
      }
      if (z < 0) {         // rounding between the lane sum and its terms
        for (int u = PER - 1; u >= 0; --u)
          if (w[u] > 0.0) { z = g0 + lane * PER + u; break; }
      } else {
        margin = fmin(tl2 - Cp, C - tl2);
      }
    }
    z = __shfl_sync(0xffffffffu, z, f);
    margin = __shfl_sync(0xffffffffu, margin, f);
  } else {
    const unsigned pos = __ballot_sync(0xffffffffu, mine > 0.0);
    if (pos) {
      const int l = 31 - __clz(pos);
      int zz = -1;
      if (lane == l)
        for (int u = PER - 1; u >= 0; --u)
          if (w[u] > 0.0) { zz = g0 + lane * PER + u; break; }
      z = __shfl_sync(0xffffffffu, zz, l);
    }
  }
  *margin_out = margin;
  return z;
}

// Extended-precision weights of one lane's PER tokens (rounds taken again
// near a tie).
template <int PER>
__device__ __forceinline__ void precise_weights(const DrawX& X, const float (&xt)[PER], const float (&xd)[PER], bool two,
                                             int t0, const float2* tab, double (&w)[PER]) {
#pragma unroll 1
  for (int u = 0; u < PER; ++u) w[u] = df_to_double(draw_weight_x(X, xt[u], two ? xd[u] : 0.f, t0 + u, tab));
}

struct DrawOut {
  int r, z;
  double margin, W;                 // margin: distance of t from the drawn bucket's nearer edge
};

// One round of the draw (DK_RESID, DK_P, DK_PRESID), once its slices are
// summed (warp-wide): locate_draw, then the token from the group's weights
// recomputed by the owner (one 16-byte load per lane and row, from L2 when
// the rows are 16-byte aligned): fp32 residual weights for DK_RESID (the
// rounding order of the consumers' slice sums), extended-precision weights
// otherwise.
template <int DT>
__device__ DrawOut draw_round(const Params& P, int b, int k, const DrawX& X, const RowStats& tr, const RowStats& dr,
                              float c, float ud, unsigned tag, const float2* tab, int lane) {
  constexpr int N = VecT<DT>::N;
  constexpr int PER = N;                             // tokens per lane in the walk
  DrawOut o{DR_FAIL, -1, 0.0, 0.0};
  const DrawLoc L = locate_draw<DT>(P, b, ud, tag, lane);
  o.r = L.r;
  o.W = L.W;
  if (L.r != DR_OK) return o;
  const int G = P.G, V = P.V, e1 = min(L.e0 + stage_elems(DT), V);
  const bool two = X.kind != DK_P && X.kind != DK_PF;
  const long long trow = row_elem_offset(KIND_TARGET, b, k, G, V);
  const long long drow = two ? row_elem_offset(KIND_DRAFT, b, k, G, V) : 0;
  const int t0 = L.g0 + lane * PER;
  float xt[PER], xd[PER];
  if (P.aligned_rows && t0 + PER <= e1) {
    constexpr int ES = DT == SPEC_BF16 ? 2 : 4;
    VecT<DT>::unpack(__ldg(reinterpret_cast<const uint4*>(P.target + (size_t)(trow + t0) * ES)), xt);
    if (two) VecT<DT>::unpack(__ldg(reinterpret_cast<const uint4*>(P.draft + (size_t)(drow + t0) * ES)), xd);
  } else {
#pragma unroll
    for (int u = 0; u < PER; ++u) {
      const int e = t0 + u;
      xt[u] = e < e1 ? load_logit(P.target, DT, trow + e) : -INFINITY;
      xd[u] = (two && e < e1) ? load_logit(P.draft, DT, drow + e) : -INFINITY;
    }
  }
  double w[PER];
  if (X.kind == DK_RESID) {
    ResidW R;
    R.c = c; R.ks = scale_k(c, X.k_lo); R.mpc = ref_of(tr.m, c); R.mqc = ref_of(dr.m, c); R.rp = 1.f / tr.s; R.nrq = -1.f / dr.s;
#pragma unroll
    for (int u = 0; u < PER; ++u) w[u] = (double)R(xt[u], xd[u]);
  } else if (X.kind == DK_PF) {
    const PW Wp{c, scale_k(c, X.k_lo), ref_of(tr.m, c)};
#pragma unroll
    for (int u = 0; u < PER; ++u) w[u] = t0 + u == X.excl ? 0.0 : (double)Wp(xt[u]);
  } else {
    precise_weights<PER>(X, xt, xd, two, t0, tab, w);
  }
  o.z = walk_group<PER>(w, L.g0, L.tl2, &o.margin, lane);
  o.r = o.z >= 0 ? DR_OK : DR_FAIL;
  return o;
}

// The round of extended-precision row sums (DK_SUMS): S_p and S_q summed
// over the slices in order (fp64).  Warp-wide; false if the wait gave up.
__device__ bool draw_sums(const Params& P, int b, unsigned tag, int lane, double* Sp, double* Sq) {
  if (!wait_slices(P, b, tag, 4, lane)) return false;
  const tword* sums = P.dsum + (size_t)kSliceWords * b * P.nres;
  double a = 0.0, q = 0.0;
  for (int j0 = 0; j0 < P.nres; j0 += 32) {
    const int j = j0 + lane;
    const double va = j < P.nres ? tagged_f64(sums, kSliceWords * j) : 0.0;
    const double vq = j < P.nres ? tagged_f64(sums, kSliceWords * j + 2) : 0.0;
    const double ia = warp_incl_scan(va, lane), iq = warp_incl_scan(vq, lane);
    a += __shfl_sync(0xffffffffu, ia, 31);
    q += __shfl_sync(0xffffffffu, iq, 31);
  }
  *Sp = a;
  *Sq = q;
  return true;
}

// 1 / S as hi + lo fp32 (S in fp64)
__device__ __forceinline__ DF recip_df(double S) {
  const double r = 1.0 / S;
  const float hi = (float)r;
  return DF{hi, (float)(r - (double)hi)};
}

// The rounds of a draw after its first (near a tie, or zero residual mass):
// extended precision, then p_k itself after zero mass.  Updates *out and
// *st; returns true if a wait gave up.
template <int DT>
__device__ __forceinline__ bool retake_draw(const Params& P, int b, int k, DrawX X, const RowStats& tr, const RowStats& dr,
                                         float c, float ud, unsigned epoch, const float2* tab, int lane, int* st,
                                         DrawOut* out) {
  DrawOut o = *out;
  int round = 0;
  if (X.kind == DK_PF && o.r != DR_FAIL && (o.r == DR_ZERO || !(o.margin >= (double)kDrawGuard * o.W))) {
    *st |= SPEC_ST_GUARDED;
    if (lane == 0) atomicAdd(&HDR_UNCERTAIN(P.hdr), 1u);
    X.kind = DK_P;
    start_draw(P, b, k, X, tr, dr, c, ++round, epoch, lane);
    o = draw_round<DT>(P, b, k, X, tr, dr, c, ud, draw_tag(epoch, round), tab, lane);
  } else if (X.kind == DK_RESID && o.r != DR_FAIL && (o.r == DR_ZERO || !(o.margin >= (double)kDrawGuard * o.W))) {
    *st |= SPEC_ST_GUARDED;
    if (lane == 0) atomicAdd(&HDR_UNCERTAIN(P.hdr), 1u);
    X.kind = DK_SUMS;
    start_draw(P, b, k, X, tr, dr, c, ++round, epoch, lane);
    double Sp = 0.0, Sq = 0.0;
    if (!draw_sums(P, b, draw_tag(epoch, round), lane, &Sp, &Sq)) return true;
    X.kind = DK_PRESID;
    X.r1 = recip_df(Sp);
    X.r2 = recip_df(Sq);
    start_draw(P, b, k, X, tr, dr, c, ++round, epoch, lane);
    o = draw_round<DT>(P, b, k, X, tr, dr, c, ud, draw_tag(epoch, round), tab, lane);
  }
  if (o.r == DR_ZERO && (X.kind == DK_PRESID || (X.kind == DK_P && X.excl >= 0))) {
    // residual mass zero: draw from p_k itself
    *st |= SPEC_ST_ZERO_RESIDUAL;
    X.kind = DK_P;
    X.excl = -1;
    start_draw(P, b, k, X, tr, dr, c, ++round, epoch, lane);
    o = draw_round<DT>(P, b, k, X, tr, dr, c, ud, draw_tag(epoch, round), tab, lane);
  }
  *out = o;
  return false;
}

// The final draw of request b (warp-wide), once k is known.  Every draw
// first runs with fp32 weights (a residual one with the streaming row sums);
// if its token lies within kDrawGuard W of a bucket edge (or the fp32 mass
// is 0) it is taken again in extended precision (a residual: row sums S_p,
// S_q first, then the weights; see retake_draw) and the request reports
// SPEC_ST_GUARDED.  Sets *z, or error bits in *st; returns true if a wait
// gave up.
template <int DT>
__device__ __forceinline__ bool run_draw(const Params& P, int b, int k, bool rejected, const RowStats& tr,
                                      const RowStats& dr, float c, unsigned epoch, int lane, int* st, int* z) {
  const int G = P.G;
  const float clo = __ldg(P.req_scale_lo + b);
  extern __shared__ __align__(128) unsigned char smem_raw[];
  const float2* tab = reinterpret_cast<const VSmem*>(smem_raw)->exp2tab;
  const float ud = P.uniforms[(size_t)b * (G + 1) + G];
  if (!(ud >= 0.f && ud < 1.f)) {
    *st = SPEC_ST_BAD_UNIFORM;
    return false;
  }
  DrawX X;
  X.m1 = tr.m; X.m2 = dr.m; X.k_hi = c; X.k_lo = clo;
  X.r1 = X.r2 = DF{0.f, 0.f};
  X.excl = -1;
  X.kind = DK_PF;
  if (rejected && P.mode == MODE_SAMPLE) X.kind = DK_RESID;
  else if (rejected) X.excl = P.draft_tokens[(size_t)b * G + k];    // one-hot residual: p without y_k
  int round = 0;
  start_draw(P, b, k, X, tr, dr, c, round, epoch, lane);
  DrawOut o = draw_round<DT>(P, b, k, X, tr, dr, c, ud, draw_tag(epoch, round), tab, lane);
  const bool near_tie = o.r != DR_FAIL && (o.r == DR_ZERO || !(o.margin >= (double)kDrawGuard * o.W));
  if (near_tie || (o.r == DR_ZERO && X.excl >= 0)) {
    if (retake_draw<DT>(P, b, k, X, tr, dr, c, ud, epoch, tab, lane, st, &o)) return true;
  }
  if (o.r != DR_OK) return true;
  *z = o.z;
  return false;
}

// Outputs of one request (warp-wide): committed tokens y_0..y_{k-1} then z,
// accept_prob for positions <= k, the SpecKV signals (H_i = log2 s_i -
// t_i / s_i bits and c_i = max_v q_i(v), held by lane i), status; then the
// request is counted as done.
__device__ void owner_outputs(const Params& P, int b, int gam, int st, int k, int z, float a_lane, float H_lane,
                              float cf_lane, unsigned epoch, int lane) {
  const int G = P.G;
  if (st & kVoidMask) {
    write_void_outputs(P, b, st, lane, 32);
  } else {
    if (P.mode != MODE_SIGNALS) {
      for (int j = lane; j <= G; j += 32)
        P.tokens[(size_t)b * (G + 1) + j] = j < k ? P.draft_tokens[(size_t)b * G + j] : (j == k ? z : -1);
      if (P.accept_prob && lane < G)
        P.accept_prob[(size_t)b * G + lane] = (lane < gam && lane <= k) ? a_lane : qnan();
      if (lane == 0) P.accept_len[b] = k;
    }
    if (P.signals_on && (P.signals || P.row_signals)) {
      const bool in = lane < gam;
      const float H = in ? H_lane : 0.f, cf = in ? cf_lane : 0.f;
      if (P.row_signals && lane < G) {
        float* rs = P.row_signals + ((size_t)b * G + lane) * 2;
        rs[0] = in ? H : qnan();
        rs[1] = in ? cf : qnan();
      }
      float hs = H, cs = cf, hm = in ? H : -INFINITY, cm = in ? cf : INFINITY;
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        hs += __shfl_xor_sync(0xffffffffu, hs, off);
        cs += __shfl_xor_sync(0xffffffffu, cs, off);
        hm = fmaxf(hm, __shfl_xor_sync(0xffffffffu, hm, off));
        cm = fminf(cm, __shfl_xor_sync(0xffffffffu, cm, off));
      }
      if (lane == 0 && P.signals) {
        float* sg = P.signals + (size_t)b * 4;
        if (gam > 0) {
          sg[0] = hs / (float)gam; sg[1] = hm; sg[2] = cs / (float)gam; sg[3] = cm;
        } else {
          sg[0] = sg[1] = sg[2] = sg[3] = qnan();
        }
      }
    }
    if (lane == 0 && P.status) P.status[b] = st;
  }
  __syncwarp();
  if (lane == 0) {
    P.req_fin[b] = part_tag(epoch);
    atomicAdd(&P.hdr->done.v, 1u);
  }
}

// Request b from its row partials to its outputs (warp-wide).  Errors are
// taken in the method's order: positions in order, then the bonus row, then
// the draw's uniform; with signals requested, a draft row that is not
// usable voids the request (the signals are read before the positions).

template <int DT, bool GREEDY>
__device__ void serve_request(const Params& P, int b, unsigned epoch, int lane) {
  const int B = P.B, G = P.G;
  const int gam = __ldg(P.req_gam + b);
  const float c = GREEDY ? 0.f : __ldg(P.req_scale + b);
  const float ks = GREEDY ? 0.f : __ldg(P.req_ks + b);

  const bool sample = P.mode == MODE_SAMPLE;
  const bool sig = P.signals_on != 0;
  float a_lane = qnan(), H_lane = qnan(), cf_lane = qnan();
  bool sig_bad = false, failed = false, rejected = false;
  int st = 0, k = gam, z = -1, ndraft = 0;   // ndraft: draft rows merged so far (0 .. ndraft-1)
  RowRes rt{}, rd{};                          // rows k of the draw
  rd.st.m = 0.f; rd.st.s = 1.f;
  auto take_draft = [&](int i, const RowRes& D) {
    if (sig) {
      if (lane == i) {
        // H = log2 s - t/s holds for any exponent reference; the largest
        // term of s is 2^{fl(m c - R(m))}, not exactly 1, so max q is that
        // term over s
        H_lane = log2f(D.st.s) - D.st.t / D.st.s;
        cf_lane = ex2(stretch(fmaf(D.st.m, c, -ref_of(D.st.m, c)), ks)) / D.st.s;
      }
      sig_bad |= !row_ok(D.st, false);
    }
  };

  // Position i decided from its merged rows; false once the scan stops.
  auto decide = [&](int i, int y, const RowRes& T, const RowRes& D) -> bool {
    if (sample) {
      take_draft(i, D);
      ndraft = i + 1;
    }
    float a;
    const int code = evaluate_pos<GREEDY>(P, b, i, T, D, y, c, ks, &a);
    if (lane == i) a_lane = a;
    if (code & PC_UNCERTAIN) {
      if (lane == 0) atomicAdd(&HDR_UNCERTAIN(P.hdr), 1u);
    } else if (code != PC_ACCEPT && lane == 0) {
      asm volatile("st.relaxed.gpu.global.b32 [%0], %1;" ::"l"(P.known_reject + b), "r"(i) : "memory");  // early exit
    }
    if ((code & 15) == PC_ACCEPT) {
      // position i accepted: the rows lookahead positions further on are now
      // worth reading, ahead of the signal-only draft rows of other requests
      const int j = i + P.lookahead;
      if (j <= gam) enqueue_row(P, target_row_id(b, j, G), epoch, lane);
      if (sample && j < gam) enqueue_row(P, draft_row_id(b, j, B, G), epoch, lane);
      return true;
    }
    k = i;
    if ((code & 15) == PC_REJECT) { rejected = true; rt = T; rd = D; }
    else st = status_of_code(code & 15);
    return false;
  };
  // the logit of row (kind, i) at the draft token y, read by the owner
  // (NaN when y is out of range: the position is then voided as a bad token)
  auto logit_at = [&](int kind, int i, int y) -> float {
    if (GREEDY || y < 0 || y >= P.V) return qnan();
    return load_logit(kind == KIND_TARGET ? P.target : P.draft, DT, row_elem_offset(kind, b, i, G, P.V) + y);
  };
  // the draft tokens and x_y of every position, loaded once (lane i holds
  // position i; G <= 31): no step of the position loop waits on them
  int y_lane = -1;
  float xt_lane = qnan(), xd_lane = qnan();
  if (P.mode != MODE_SIGNALS && lane < gam) {
    y_lane = P.draft_tokens[(size_t)b * G + lane];
    xt_lane = logit_at(KIND_TARGET, lane, y_lane);
    if (sample) xd_lane = logit_at(KIND_DRAFT, lane, y_lane);
  }
  bool bonus = false;                         // the bonus row is merged (into rt)
  if (P.mode != MODE_SIGNALS && P.nch <= 8) {
    // position i, and position i+1 (or the bonus row) too when its rows are
    // already complete: an owner behind the stream catches up two at a time
    for (int i = 0; i < gam;) {
      const int i1 = i + 1;
      const int y0 = __shfl_sync(0xffffffffu, y_lane, i);
      const int y1 = __shfl_sync(0xffffffffu, y_lane, i1 & 31);
      const int seg = lane >> 3;
      int rid = -1;
      if (seg == 0) rid = target_row_id(b, i, G);
      else if (seg == 1) rid = sample ? draft_row_id(b, i, B, G) : -1;
      else if (seg == 2) rid = i1 <= gam ? target_row_id(b, i1, G) : -1;
      else rid = (sample && i1 < gam) ? draft_row_id(b, i1, B, G) : -1;
      // x_y of the four rows (positions i, i + 1 of target and draft)
      const float xt0 = __shfl_sync(0xffffffffu, xt_lane, i), xd0 = __shfl_sync(0xffffffffu, xd_lane, i);
      const float xt1 = __shfl_sync(0xffffffffu, xt_lane, i1 & 31), xd1 = __shfl_sync(0xffffffffu, xd_lane, i1 & 31);
      Part pm;
      const int ready = merge_rows4<GREEDY>(P, rid, (seg & 1) && sig, 3u, c, ks, epoch, lane, pm);
      if (ready < 0) { failed = true; break; }
      auto row_xy = [&](int s2) {
        RowRes o = row_of(pm, s2);
        o.xy = s2 == 0 ? xt0 : s2 == 1 ? xd0 : s2 == 2 ? xt1 : xd1;
        return o;
      };
      if (!decide(i, y0, row_xy(0), row_xy(1))) break;
      if (i1 < gam && (ready & 12) == 12) {
        if (!decide(i1, y1, row_xy(2), row_xy(3))) break;
        i += 2;
      } else {
        if (i1 == gam && (ready & 4)) { rt = row_of(pm, 2); bonus = true; }
        i += 1;
      }
    }
  } else if (P.mode != MODE_SIGNALS) {
    for (int i = 0; i < gam; ++i) {
      const int y = __shfl_sync(0xffffffffu, y_lane, i);
      RowRes T, D{};
      const float xt = __shfl_sync(0xffffffffu, xt_lane, i), xd = __shfl_sync(0xffffffffu, xd_lane, i);
      if (sample && 2 * P.nch <= 32) {
        if (!merge_pair(P, target_row_id(b, i, G), draft_row_id(b, i, B, G), c, ks, sig, epoch, lane, T, D)) {
          failed = true;
          break;
        }
      } else {
        if (!merge_row<GREEDY>(P, target_row_id(b, i, G), c, ks, false, epoch, lane, T)) {
          failed = true;
          break;
        }
        if (sample && !merge_row<false>(P, draft_row_id(b, i, B, G), c, ks, sig, epoch, lane, D)) {
          failed = true;
          break;
        }
      }
      T.xy = xt;
      D.xy = xd;
      if (!decide(i, y, T, D)) break;
    }
  }
  if (P.mode != MODE_SIGNALS && !failed && st == 0 && !rejected) {   // every position accepted: the bonus row
    if (!bonus && !merge_row<GREEDY>(P, target_row_id(b, gam, G), c, ks, false, epoch, lane, rt)) failed = true;
    else if (!row_ok(rt.st, GREEDY)) st = SPEC_ST_NONFINITE;
  }
  // the draw is started as soon as k is known, and finished before the
  // remaining signal rows are merged (they are read last)
  if (!GREEDY && P.mode != MODE_SIGNALS && !failed && st == 0)
    failed = run_draw<DT>(P, b, k, rejected, rt.st, rd.st, c, epoch, lane, &st, &z);
  // the signal rows not merged yet (they stream after the rows of the first
  // positions)
  if (sig && !failed) {
    for (int i = ndraft; i < gam;) {
      if (P.nch <= 8) {            // up to four draft rows per pass: the first waited for
        const int j = i + (lane >> 3);
        Part pm;
        const int ready = merge_rows4<false>(P, j < gam ? draft_row_id(b, j, B, G) : -1, true, 1u, c, ks, epoch, lane, pm);
        if (ready < 0) { failed = true; break; }
        int s2 = 0;
        for (; s2 < 4 && i + s2 < gam && ((ready >> s2) & 1); ++s2) take_draft(i + s2, row_of(pm, s2));
        i += s2;
      } else {
        RowRes D;
        if (!merge_row<false>(P, draft_row_id(b, i, B, G), c, ks, true, epoch, lane, D)) { failed = true; break; }
        take_draft(i, D);
        ++i;
      }
    }
  }
  if (GREEDY && !failed && st == 0) z = rt.st.idx & ~kIdxNaN;
  if (failed) st = SPEC_ST_TIMEOUT;
  else if (sig && __any_sync(0xffffffffu, sig_bad)) st = SPEC_ST_NONFINITE;
  owner_outputs(P, b, gam, st, k, z, a_lane, H_lane, cf_lane, epoch, lane);
}

template <int DT, bool GREEDY>
__device__ __forceinline__ void owner_role(const Params& P, unsigned epoch, int lane) {
  for (int b = blockIdx.x; b < P.B; b += gridDim.x) {
    if (__ldg(P.req_status + b) & kFinished) continue;    // settled by the plan kernel
    serve_request<DT, GREEDY>(P, b, epoch, lane);
  }
}

}  // namespace

template <int DT, bool GREEDY>
__global__ void __launch_bounds__(kStatsThreads, 2) verify_kernel(const __grid_constant__ Params P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  VSmem& S = *reinterpret_cast<VSmem*>(smem_raw);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.empty[s], kConsumerWarps);
    }
    for (int e = 0; e < kEpiSlots; ++e) {
      mbar_init(&S.epi_full[e], kConsumerWarps);
      mbar_init(&S.epi_empty[e], 1);
      S.slot[e].term = 0;
    }
    S.abort = 0;
    S.fifo_head = S.fifo_tail = S.prio_full = 0;
    S.wait_limit = P.wait_limit;
    fence_mbar_init();
  }
  for (int j = threadIdx.x; j < 256; j += blockDim.x) S.exp2tab[j] = kExp2Tab[j];
  __syncthreads();
  griddep_wait();   // the plan kernel's schedule, counters and epoch are ready
  const unsigned epoch = HDR_EPOCH(P.hdr);   // partials and queue entries carry 8 * epoch
  if (warp < kConsumerWarps) consumer_role<DT, GREEDY>(P, S, warp, lane);
  else if (warp == kConsumerWarps) {
    if (lane == 0) producer_role<DT, GREEDY>(P, S);
  } else if (warp <= kConsumerWarps + kEpiWarps) {
    epilogue_role<DT, GREEDY>(P, S, lane, warp - kConsumerWarps - 1, epoch);
  } else if (warp == kConsumerWarps + kEpiWarps + 1) {
    if (lane == 0) scheduler_role<DT, GREEDY>(P, S, epoch);
  } else {
    owner_role<DT, GREEDY>(P, epoch, lane);
  }
  __syncthreads();
  // the last CTA out voids any request an aborted wait left unfinished
  if (threadIdx.x == 0) {
    __threadfence();
    const unsigned ex = atomicAdd(&HDR_EXITED(P.hdr), 1u) + 1u;
    if (ex == gridDim.x && ld_relaxed_u32(&P.hdr->error.v) != 0u) {
      __threadfence();
      for (int b = 0; b < P.B; ++b)
        if (!(__ldcg(P.req_status + b) & kFinished) && __ldcg(P.req_fin + b) != part_tag(epoch))
          write_void_outputs(P, b, SPEC_ST_TIMEOUT, 0, 1);
    }
  }
}

static size_t verify_smem_bytes() { return sizeof(VSmem); }

cudaError_t configure_kernels() {
  const int smem = (int)verify_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(verify_kernel<SPEC_F32, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(verify_kernel<SPEC_F32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(verify_kernel<SPEC_BF16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(verify_kernel<SPEC_BF16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return e;
}

// Resident CTAs per SM of the verify kernel (the least over its
// instantiations).  The kernel is persistent and its CTAs wait on one
// another, so its grid never exceeds what is resident at once.
cudaError_t verify_blocks_per_sm(int* out) {
  void (*ks[4])(const Params) = {verify_kernel<SPEC_F32, false>, verify_kernel<SPEC_F32, true>,
                           verify_kernel<SPEC_BF16, false>, verify_kernel<SPEC_BF16, true>};
  int best = 1 << 30;
  for (auto k : ks) {
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, kStatsThreads, verify_smem_bytes());
    if (e != cudaSuccess) return e;
    best = n < best ? n : best;
  }
  *out = best;
  return cudaSuccess;
}

cudaError_t launch_plan(const Params& P, cudaStream_t s) {
  return launch_ex(plan_kernel, dim3(1), dim3(1024), 0, s, false, P);
}

cudaError_t launch_verify(const Params& P, int grid, cudaStream_t s, bool pdl) {
  const bool greedy = P.mode == MODE_GREEDY;
  void (*k)(const Params) = P.dtype == SPEC_BF16 ? (greedy ? verify_kernel<SPEC_BF16, true> : verify_kernel<SPEC_BF16, false>)
                                           : (greedy ? verify_kernel<SPEC_F32, true> : verify_kernel<SPEC_F32, false>);
  return launch_ex(k, dim3(grid), dim3(kStatsThreads), verify_smem_bytes(), s, pdl, P);
}

}  // namespace sv
