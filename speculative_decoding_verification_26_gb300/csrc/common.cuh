// common.cuh -- shared definitions of the sm_103a verification kernels:
// launch parameters, workspace layout, inline-PTX wrappers (mbarrier, bulk
// copy, scoped atomics) and the per-row softmax statistics.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/spec_verify.h"

namespace sv {

// ---------------------------------------------------------------------------
// modes and codes

enum Mode : int { MODE_GREEDY = 0, MODE_SAMPLE = 1, MODE_ONEHOT = 2, MODE_SIGNALS = 3 };
enum RowKind : int { KIND_TARGET = 0, KIND_DRAFT = 1 };

// per-position test result written by the stats kernel, read by finalize
enum PairCode : int {
  PC_NONE = 0,        // not evaluated (position after a known reject)
  PC_ACCEPT = 1,
  PC_REJECT = 2,
  PC_NONFINITE = 3,
  PC_BAD_TOKEN = 4,
  PC_BAD_UNIFORM = 5,
};
constexpr int PC_UNCERTAIN = 16;   // or-ed in: |u - a| inside the guard band

// work items of the persistent kernel
enum ItemType : int {
  IT_STATS = 1,    // 64 KB chunk of one logit row: softmax statistics
  IT_DSUM = 2,     // one 16 KB slice of the draw's weights: group sums
};

// draw kinds (one round of a draw each):
//   DK_RESID   the residual [p_k - q_k]_+ (rows k of both models) with fp32
//              weights and the streaming row sums;
//   DK_P       2^{a} of target row k in extended precision (bonus draw;
//              one-hot residual with the draft token removed);
//   DK_SUMS    the extended-precision row sums S_p, S_q of rows k (first
//              round of a residual draw taken again in extended precision);
//   DK_PRESID  [p_k - q_k]_+ in extended precision with S_p, S_q from DK_SUMS;
//   DK_PF      2^{a} of target row k with fp32 weights (first round of a
//              bonus or one-hot draw; taken again as DK_P near a tie).
enum DrawKind : int { DK_RESID = 1, DK_P = 2, DK_SUMS = 3, DK_PRESID = 4, DK_PF = 5 };
constexpr int kMaxDrawRounds = 4;   // residual, sums, extended residual, p after zero mass


// ---------------------------------------------------------------------------
// geometry

constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kEpiWarps = 1;                           // epilogue warps (items alternate)
constexpr int kStatsThreads = kConsumerThreads + 32 * (3 + kEpiWarps);   // + producer, scheduler, epilogue, owner warps
constexpr int kStageBytes = 16384;                      // one bulk copy
constexpr int kStages = 4;                              // ring depth per CTA
constexpr int kChunkBytes = 4 * kStageBytes;            // one work item of a row
constexpr int kEpiSlots = 12;                           // consumer -> epilogue ring (multiple of kEpiWarps)
constexpr int kGroupVecs = 32;                          // draw group: one warp's 32 vectors (256 bf16 / 128 fp32 tokens)
constexpr int kGroupsPerStage = kStageBytes / 16 / kGroupVecs;   // 32
constexpr int kPartWords = 3;                           // tagged words of a chunk partial: m, s (argmax: idx), t
constexpr int kDrawWords = 12;                          // tagged words of a draw descriptor
constexpr int kSliceWords = 4;                          // tagged words of a draw slice's sums (two fp64)
constexpr int kGroupWords = 2;                          // tagged words of a draw group sum (one fp64)
constexpr int kNoReject = 0x7fffffff;
constexpr unsigned kEpochMax = 0x1ffffff0u;             // tags come from 8 * epoch + kind (kind < 8)
// Tags are (8 * epoch + kind) * kTagMul: an odd multiplier is a bijection of
// the 32-bit integers that maps 0 to 0 only, and sends the small integers an
// epoch starts from to values that stale data (counts, indices, tokens) does
// not hold.
constexpr unsigned kTagMul = 0x9E3779B1u;
constexpr unsigned long long kWorkspaceMagic = 0x5356455246595631ull;
// Every bounded wait counts SM clock cycles (clock64 is a register of the SM
// and costs a few cycles to read; the global timer is read from outside the
// SM and delays the reading warp by about a microsecond under load).
// 4e9 cycles: about 2 s at the maximum clock, longer when clocked down.  The
// limit of a call is Params::wait_limit (this default unless a test lowers
// it); the wait for a CTA's own bulk copies still in flight before it exits
// always uses the default, so no copy can land in shared memory after exit.
constexpr long long kWaitLimitCycles = 4000000000ll;

// ---------------------------------------------------------------------------
// partial statistics of a run of logits, relative to the exponent reference
// R(m) = fl(m c) of its own max m (see ref_of), with a = stretch(fl(x c - R(m)), k):
//   s = sum 2^a,  t = sum a 2^a  (entropy numerator),
//   idx = lowest index attaining m,  bad = a NaN was seen (argmax mode).
struct alignas(16) Part {
  float m, s, t;
  int idx;   // bit 30 set: NaN seen (argmax mode); low bits: index
};
constexpr int kIdxNaN = 1 << 30;

struct alignas(16) RowStats {
  float m, s, t;
  int idx;
};

// ---------------------------------------------------------------------------
// workspace layout (offsets in bytes, 256-aligned)

struct Layout {
  size_t hdr, req_flags, known_reject, row_list, req_scale, req_scale_lo, req_ks, req_gam, req_status, req_fin, cparts,
      dsum, gsum, dd, dq, claim, defq, total;
  int nrows;      // B*(G+1) + B*G row ids
  int nch;        // statistics chunks per row
  int nres;       // draw slices per row (one stage each)
  int dq_cap;     // dynamic queue capacity: every draw round and lookahead row
  int def_cap;    // deferred queue capacity (statistics items of draft rows)
};

// Counters of one call, each on its own 128-byte line: they are hit by
// atomics from every CTA, and sharing a line would serialise unrelated ones.
struct alignas(128) Counter {
  unsigned int v;
  unsigned int pad[31];
};

struct Header {
  Counter queue;        // next static (statistics) item to claim
  Counter dq_head;      // next dynamic-queue ticket
  Counter dq_tail;      // dynamic items reserved
  Counter def_head;     // next deferred-queue ticket
  Counter def_tail;     // deferred static items reserved
  Counter done;         // requests whose outputs are written
  Counter error;        // SPEC_ST_TIMEOUT when any wait gave up
  Counter misc;         // n_items, n_valid, exited, n_uncertain, epoch, n_front, magic, generation, owner (rarely written)
};
#define HDR_N_ITEMS(h) ((h)->misc.pad[0])
#define HDR_N_VALID(h) ((h)->misc.pad[1])
#define HDR_EXITED(h) ((h)->misc.pad[2])
#define HDR_UNCERTAIN(h) ((h)->misc.pad[3])
#define HDR_EPOCH(h) ((h)->misc.pad[4])
#define HDR_N_FRONT(h) ((h)->misc.pad[5])   // static items of the first positions
#define HDR_MAGIC(h) (*reinterpret_cast<unsigned long long*>(&(h)->misc.pad[7]))   // byte offset 32: 8-aligned
#define HDR_GEN(h) (*reinterpret_cast<unsigned long long*>(&(h)->misc.pad[9]))     // byte offset 40: 8-aligned
// the address of the call counter of the library copy that last used the
// workspace (two copies of the library in one process count calls apart)
#define HDR_OWNER(h) (*reinterpret_cast<unsigned long long*>(&(h)->misc.pad[11]))   // byte offset 48: 8-aligned

// Data that crosses CTAs travels in tagged 64-bit words: payload in the high
// 32 bits, the tag in the low 32 bits: (8 * epoch) * kTagMul for chunk
// partials and queue entries, (8 * epoch + 1 + round) * kTagMul for the words
// of a draw round (one tag space per kind of word).  An aligned 64-bit
// relaxed access is single-copy atomic, so a reader that sees the current tag
// has the payload written in this call, whatever the order in which words
// become visible: no fence and no counter is needed to publish them.  Every
// call on the device has its own epoch (one counter for all workspaces), so
// words left by earlier calls, in this workspace or in memory another
// workspace or tensor held before, are not mistaken for new ones.
typedef unsigned long long tword;

__host__ __device__ inline size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

__host__ __device__ inline int chunk_elems(int dtype) { return kChunkBytes / (dtype == SPEC_BF16 ? 2 : 4); }
__host__ __device__ inline int stage_elems(int dtype) { return kStageBytes / (dtype == SPEC_BF16 ? 2 : 4); }

__host__ inline Layout make_layout(int B, int G, int V, int dtype) {
  Layout L{};
  const int nrows = B * (G + 1) + B * G;
  const int ce = chunk_elems(dtype), se = stage_elems(dtype);
  L.nrows = nrows;
  L.nch = (V + ce - 1) / ce;
  L.nres = (V + se - 1) / se;
  // every round of every draw, and the chunks of every lookahead row (target
  // rows 2..G and, without signals, draft rows 2..G-1 of each request)
  L.dq_cap = B * (kMaxDrawRounds * L.nres + 2 * G * L.nch + 2);
  L.def_cap = B * G * L.nch;
  size_t o = 0;
  L.hdr = o;          o = align256(o + sizeof(Header));
  L.req_flags = o;    o = align256(o + sizeof(int) * B);
  L.known_reject = o; o = align256(o + sizeof(int) * B);
  L.row_list = o;     o = align256(o + sizeof(int) * nrows);
  L.req_scale = o;    o = align256(o + sizeof(float) * B);
  L.req_scale_lo = o; o = align256(o + sizeof(float) * B);
  L.req_ks = o;       o = align256(o + sizeof(float) * B);
  L.req_gam = o;      o = align256(o + sizeof(int) * B);
  L.req_status = o;   o = align256(o + sizeof(int) * B);
  L.req_fin = o;      o = align256(o + sizeof(unsigned) * B);
  L.cparts = o;       o = align256(o + sizeof(tword) * (size_t)nrows * L.nch * kPartWords);
  L.dsum = o;         o = align256(o + sizeof(tword) * kSliceWords * (size_t)B * L.nres);
  L.gsum = o;         o = align256(o + sizeof(tword) * (size_t)B * L.nres * kGroupsPerStage * kGroupWords);
  L.dd = o;           o = align256(o + sizeof(tword) * kDrawWords * (size_t)B);
  L.dq = o;           o = align256(o + sizeof(tword) * 2 * (size_t)L.dq_cap);
  L.claim = o;        o = align256(o + sizeof(tword) * (size_t)B * G * L.nch);
  L.defq = o;         o = align256(o + sizeof(tword) * (size_t)L.def_cap);
  L.total = o;
  return L;
}

// ---------------------------------------------------------------------------
// launch parameters (passed by value to every kernel)

struct Params {
  const unsigned char* target;   // [B, G+1, V]
  const unsigned char* draft;    // [B, G, V] or null
  int dtype, B, G, V, mode, signals_on;
  int aligned_rows;              // every row starts on a 16-byte boundary
  int keep_pos;                  // rows of positions <= keep_pos are kept in L2 for the draw (-1: none)
  long long wait_limit;          // SM cycles before a wait gives up (kWaitLimitCycles unless lowered)
  const int32_t* draft_tokens;
  const int32_t* gamma;
  const float* temperature;
  const float* uniforms;
  int32_t* accept_len;
  int32_t* tokens;
  int32_t* status;
  float* signals;
  float* row_signals;
  float* accept_prob;
  // workspace views
  Header* hdr;
  int* req_flags;                // error bits found by the plan kernel
  int* known_reject;             // earliest decided reject (early exit), relaxed
  int* row_list;                 // position-major row schedule
  float* req_scale;              // log2(e) / T_b rounded to fp32 (plan kernel)
  float* req_scale_lo;           // log2(e) / T_b - req_scale, rounded to fp32 (extended-precision draws)
  float* req_ks;                 // scale_k(req_scale, req_scale_lo): the exponent stretch (see ref_of)
  int* req_gam;                  // gamma_b (plan kernel)
  int* req_status;               // kFinished: settled by the plan kernel
  unsigned* req_fin;             // tag of the call whose outputs were written
  tword* cparts;                 // [nrows][nch][kPartWords] chunk partials
  tword* dsum;                   // [B][nres][kSliceWords] draw slice sums (one or two fp64 as hi, lo words)
  tword* gsum;                   // [B][nres][kGroupsPerStage][kGroupWords] draw group sums (fp64)
  tword* dd;                     // [B][kDrawWords] draw descriptors
  tword* dq;                     // [dq_cap][2] dynamic work queue (draw slices, lookahead row chunks)
  tword* claim;                  // [B][G][nch] draft-row chunks taken (a static item and a lookahead entry race for them)
  tword* defq;                   // [def_cap] deferred static items (main-queue index): signal-only draft rows
  int nrows, nch, nres, dq_cap, def_cap;
  int lookahead;                 // target rows of positions >= lookahead are read once position - lookahead is accepted
};

// row ids: target rows first, then draft rows
__host__ __device__ inline int target_row_id(int b, int i, int G) { return b * (G + 1) + i; }
__host__ __device__ inline int draft_row_id(int b, int i, int B, int G) { return B * (G + 1) + b * G + i; }

__device__ inline void decode_row(int rid, int B, int G, int& kind, int& b, int& i) {
  const int nt = B * (G + 1);
  if (rid < nt) { kind = KIND_TARGET; b = rid / (G + 1); i = rid - b * (G + 1); }
  else { rid -= nt; kind = KIND_DRAFT; b = rid / G; i = rid - b * G; }
}

// flat element offset of a row inside its tensor
__device__ inline long long row_elem_offset(int kind, int b, int i, int G, int V) {
  return kind == KIND_TARGET ? ((long long)b * (G + 1) + i) * V : ((long long)b * G + i) * V;
}

// ---------------------------------------------------------------------------
// inline PTX

__device__ __forceinline__ float ex2(float x) {   // 2^x, hardware approximation, ftz
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ unsigned long long globaltimer() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// As mbar_try_wait, but the thread may sleep in hardware until the phase
// completes or `hint_ns` pass (instead of returning at once): a waiting warp
// then takes no issue slots and no shared-memory bandwidth from the others.
__device__ __forceinline__ bool mbar_try_wait_sleep(uint64_t* bar, uint32_t parity, uint32_t hint_ns) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
      : "memory");
  return ok != 0;
}

// 1-D bulk copy global -> shared, completion counted on `bar` (bytes % 16 == 0,
// both addresses 16-byte aligned).
// L2 policies of the bulk copies: rows the draw may read again stay in L2
// (evict_last), the rest of the stream leaves first (evict_first).
__device__ __forceinline__ uint64_t l2_policy(bool keep) {
  uint64_t pol;
  if (keep) asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  else asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// As bulk_load, with an L2 cache policy.
__device__ __forceinline__ void bulk_load_hint(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar,
                                               uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::
          "r"(smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gmem_src, uint32_t bytes, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(smem_dst)),
      "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}



__device__ __forceinline__ int ld_relaxed(const int* p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// tagged words (see tword)
__device__ __forceinline__ tword tw_make(unsigned payload, unsigned tag) {
  return ((tword)payload << 32) | (tword)tag;
}
__device__ __forceinline__ bool tw_ok(tword w, unsigned tag) { return (unsigned)w == tag; }
__device__ __forceinline__ unsigned tw_u32(tword w) { return (unsigned)(w >> 32); }
__device__ __forceinline__ float tw_f32(tword w) { return __uint_as_float((unsigned)(w >> 32)); }
__device__ __forceinline__ tword ld_tw(const tword* p) {
  tword v;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_tw(tword* p, tword v) {
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(v) : "memory");
}

__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------------------
// logits

__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// One logit from global memory (for the few scalar accesses).
__device__ __forceinline__ float load_logit(const unsigned char* base, int dtype, long long elem) {
  if (dtype == SPEC_BF16) {
    unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(base) + elem);
    return __uint_as_float(static_cast<uint32_t>(h) << 16);
  }
  return __ldg(reinterpret_cast<const float*>(base) + elem);
}

// log2(e) / T rounded toward zero to fp32 (the scale used by every kernel;
// the remainder, >= 0, is carried separately: see ref_of)
__device__ __forceinline__ float scale_of(float T) { return __double2float_rz(1.4426950408889634 / (double)T); }

__device__ __forceinline__ bool temperature_ok(float T) { return T > 0.f && isfinite(T); }

// A row is usable iff its max is finite, its sum is finite and positive and
// no NaN was seen.
__device__ __forceinline__ bool row_ok(const RowStats& r, bool argmax_mode) {
  if (!isfinite(r.m)) return false;
  if (argmax_mode) return (r.idx & kIdxNaN) == 0;
  return isfinite(r.s) && r.s > 0.f;
}

// The exponent reference of a run of logits with max m at scale c: every
// term of its sums is 2^a with a = fl(a0 + a0 k), a0 = fl(x c - R(m)),
// R(m) = fl(m c).  c is log2(e) / T rounded toward zero to fp32 and
// c (1 + k) = c + c_lo is that scale to about 48 bits: a0 (1 + k) =
// x (c + c_lo) - R(m) (1 + k), so k corrects the fp32 rounding of c (which
// would otherwise temper every row by up to 1e-7 of its exponents) up to a
// constant of the row.  Every rescale between two runs uses
// d (1 + k), d = R(m1) - R(m2).  So all sums of a row, the probability of one
// token and the draw weights refer to the same reference of the row max (a
// common offset of every exponent of the row, which cancels in every ratio)
// and do not depend on how m c rounds (at |m c| ~ 500, half an ulp of m c is
// 3e-5 in the exponent).  k > 0, so a logit of -inf keeps the exponent -inf.
__device__ __forceinline__ float ref_of(float m, float c) { return __fmul_rn(m, c); }
__device__ __forceinline__ float scale_k(float c, float c_lo) {
  return c > 0.f ? fmaxf(__fdiv_rn(c_lo, c), 1e-30f) : 0.f;
}
__device__ __forceinline__ float stretch(float a, float k) { return __fmaf_rn(a, k, a); }

// Merge of two partials of the same row (online-softmax rule):
//   m = max(m1, m2); s = sum_j s_j 2^{d_j}, d_j = (R(m_j) - R(m)) (1 + k);
//   t = sum_j 2^{d_j}(t_j + d_j s_j).
__device__ __forceinline__ Part merge_parts(const Part& a, const Part& b, float c, float k, bool ent) {
  Part r;
  const float m = fmaxf(a.m, b.m);
  r.m = m;
  if (m == -INFINITY) {          // both empty
    r.s = 0.f; r.t = 0.f;
  } else {
    const float rm = ref_of(m, c);
    float sa = 0.f, ta = 0.f, sb = 0.f, tb = 0.f;
    if (a.s != 0.f) {
      const float d = stretch(__fsub_rn(ref_of(a.m, c), rm), k);
      const float f = ex2(d);
      sa = a.s * f;
      if (ent) ta = f * fmaf(d, a.s, a.t);
    }
    if (b.s != 0.f) {
      const float d = stretch(__fsub_rn(ref_of(b.m, c), rm), k);
      const float f = ex2(d);
      sb = b.s * f;
      if (ent) tb = f * fmaf(d, b.s, b.t);
    }
    // NaN partial sums stay NaN (the row is then rejected as non-finite)
    if (a.s != a.s) sa = a.s;
    if (b.s != b.s) sb = b.s;
    r.s = sa + sb;
    r.t = ta + tb;
  }
  const int ia = a.idx & ~kIdxNaN, ib = b.idx & ~kIdxNaN;
  int idx;
  if (a.m > b.m) idx = ia;
  else if (b.m > a.m) idx = ib;
  else idx = ia < ib ? ia : ib;
  r.idx = idx | ((a.idx | b.idx) & kIdxNaN);
  return r;
}

__device__ __forceinline__ Part shfl_part(const Part& p, int src_lane_xor) {
  Part q;
  q.m = __shfl_xor_sync(0xffffffffu, p.m, src_lane_xor);
  q.s = __shfl_xor_sync(0xffffffffu, p.s, src_lane_xor);
  q.t = __shfl_xor_sync(0xffffffffu, p.t, src_lane_xor);
  q.idx = __shfl_xor_sync(0xffffffffu, p.idx, src_lane_xor);
  return q;
}

// Merge of two argmax-only partials (greedy rows).
__device__ __forceinline__ Part merge_argmax(const Part& a, const Part& b) {
  Part r;
  r.m = fmaxf(a.m, b.m);
  r.s = 0.f; r.t = 0.f;
  const int ia = a.idx & ~kIdxNaN, ib = b.idx & ~kIdxNaN;
  int idx;
  if (a.m > b.m) idx = ia;
  else if (b.m > a.m) idx = ib;
  else idx = ia < ib ? ia : ib;
  r.idx = idx | ((a.idx | b.idx) & kIdxNaN);
  return r;
}

// 16-byte loads/stores that bypass L1 (data written by other CTAs of the grid)
__device__ __forceinline__ Part ldcg_part(const Part* p) {
  const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
  Part r;
  r.m = v.x; r.s = v.y; r.t = v.z; r.idx = __float_as_int(v.w);
  return r;
}
__device__ __forceinline__ RowStats ldcg_stats(const RowStats* p) {
  const float4 v = __ldcg(reinterpret_cast<const float4*>(p));
  RowStats r;
  r.m = v.x; r.s = v.y; r.t = v.z; r.idx = __float_as_int(v.w);
  return r;
}
__device__ __forceinline__ void stcg_part(Part* p, const Part& v) {
  __stcg(reinterpret_cast<float4*>(p), make_float4(v.m, v.s, v.t, __int_as_float(v.idx)));
}

__device__ __forceinline__ Part empty_part() {
  Part p;
  p.m = -INFINITY; p.s = 0.f; p.t = 0.f; p.idx = 0x3fffffff;
  return p;
}

// Host-side launchers (defined in verify.cu).  `pdl` enables programmatic
// dependent launch on the caller's stream.
// Parameters of the divergence-statistics kernel (divergence.cu).
struct DivParams {
  const unsigned char* target;   // [B, G+1, V]
  const unsigned char* draft;    // [B, G, V]
  int dtype, B, G, V;
  int aligned;                   // every row starts on a 16-byte boundary (vector loads)
  const int32_t* gamma;          // [B] or null (= G)
  const float* temperature;      // [B]
  float* stats;                  // [B, G, 5]
  int32_t* status;               // [B] or null (zeroed by the host before the launch)
};
cudaError_t launch_divergence(const DivParams& P, int grid, cudaStream_t s);

// Parameters of the top-k / top-p filter (filter.cu).
struct FiltParams {
  unsigned char* logits;         // [n, V], filtered in place
  int dtype, n, V;
  const int32_t* top_k;          // [n] or null
  const float* top_p;            // [n] or null
  const float* temperature;      // [n] or null (= 1)
  int32_t* status;               // [n] or null
};
cudaError_t launch_filter(const FiltParams& P, int grid, cudaStream_t s);

// The SpecKV gamma selector (gamma.cu): model of SPEC_GAMMA_MODEL_FLOATS values.
constexpr int kGammaModelFloats = SPEC_GAMMA_MODEL_FLOATS;
cudaError_t launch_gamma_select(const float* signals, const float* comp, const float* model, int B,
                                int32_t* gamma_star, float* expected, cudaStream_t s);

cudaError_t launch_plan(const Params& P, cudaStream_t s);
cudaError_t launch_verify(const Params& P, int grid, cudaStream_t s, bool pdl);
cudaError_t configure_kernels();   // dynamic shared-memory limit, current device
cudaError_t verify_blocks_per_sm(int* out);   // resident verify CTAs per SM, current device

template <class K>
inline cudaError_t launch_ex(K kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s, bool pdl, const Params& P) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = pdl ? attr : nullptr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kern, P);
}

}  // namespace sv
