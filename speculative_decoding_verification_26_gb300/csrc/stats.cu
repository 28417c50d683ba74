// stats.cu -- the row schedule (plan_kernel) and the streaming row-statistics
// kernel (stats_kernel) of the verification path.
//
// stats_kernel is a persistent, warp-specialised kernel (2 CTAs per SM):
//   * producer warp: claims work items (32 KB chunks of logit rows) from a
//     global queue in the plan's position-major order, skips rows that an
//     earlier reject has made void, and stages each chunk into a 6-deep ring
//     of 16 KB shared-memory buffers with 1-D bulk copies (cp.async.bulk)
//     completed on mbarriers;
//   * 8 consumer warps: read the staged bytes with 128-bit shared loads and
//     keep, per thread, the online softmax statistics of the run (max m,
//     s = sum 2^{(x-m)c}, and for draft rows that feed the signals
//     t = sum (x-m)c 2^{(x-m)c}); greedy rows keep the max and its lowest index;
//   * epilogue warp: merges the 8 warp partials of a chunk, publishes it, and
//     the CTA that completes a row (last arrival on the row counter) merges
//     the row's chunks in chunk order; the one that completes a position pair
//     evaluates the acceptance test of that position (tutorial page
//     "5.1 投机解码核心原理", sections 3.1-3.3) and publishes the first reject
//     so later rows of that request are skipped (section 5.1).
// Every spin is bounded in time; a wait that gives up sets SPEC_ST_TIMEOUT.
#include "common.cuh"

namespace sv {

// ---------------------------------------------------------------------------
// plan: reset the counters and build the compacted row schedule

namespace {

enum BlockType : int { BT_T = 0, BT_D = 1, BT_PAIR = 2 };

struct Block {
  int type, i;
};

// Schedule blocks in position-major order.  Full-q with signals reads every
// draft row anyway, so draft blocks are used as filler between target
// positions: PAIR(0) | D1 D2 | T1 | D3 D4 | T2 | ... | T_G.  Between the
// target rows of positions i-1 and i there are then about 2B rows of other
// work, longer than the reading window of the whole GPU, so the test at i-1
// is usually decided before target row i of the request is claimed.  Draft
// block j always precedes target block j, as the test at j needs both.
__device__ inline int build_blocks(int mode, int signals_on, int G, Block* out) {
  int n = 0;
  if (mode == MODE_SIGNALS) {
    for (int i = 0; i < G; ++i) out[n++] = {BT_D, i};
  } else if (mode == MODE_SAMPLE && signals_on && G > 0) {
    out[n++] = {BT_PAIR, 0};
    int dnext = 1;
    for (int i = 1; i <= G; ++i) {
      for (int f = 0; f < 2 && dnext <= G - 1; ++f) out[n++] = {BT_D, dnext++};
      out[n++] = {BT_T, i};
    }
  } else if (mode == MODE_SAMPLE) {
    for (int i = 0; i <= G; ++i) out[n++] = {BT_PAIR, i};
  } else {
    for (int i = 0; i <= G; ++i) out[n++] = {BT_T, i};
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

__global__ void __launch_bounds__(1024) plan_kernel(Params P) {
  griddep_launch();
  const int B = P.B, G = P.G, tid = threadIdx.x, nth = blockDim.x;
  const int lane = tid & 31, warp = tid >> 5, nwarps = nth >> 5;
  __shared__ int s_count[64];
  __shared__ int s_off[65];
  __shared__ Block s_blk[64];
  __shared__ int s_nb;

  for (int j = tid; j < P.nrows; j += nth) {
    P.row_arr[j] = 0u;
    P.row_done[j] = 0;
  }
  for (int j = tid; j < B * (G + 1); j += nth) {
    P.pair_arr[j] = 0u;
    P.pair_res[j] = PC_NONE;
    P.pair_a[j] = __longlong_as_double(0x7ff8000000000000ll);
  }
  for (int b = tid; b < B; b += nth) {
    P.known_reject[b] = kNoReject;
    P.draw_arr[b] = 0u;
    int st = 0;
    const int gam = P.gamma ? P.gamma[b] : G;
    if (gam < 0 || gam > G) st |= SPEC_ST_BAD_GAMMA;
    if (P.mode != MODE_GREEDY && !temperature_ok(P.temperature[b])) st |= SPEC_ST_BAD_TEMPERATURE;
    P.req_flags[b] = st;
  }
  if (tid == 0) s_nb = build_blocks(P.mode, P.signals_on, G, s_blk);
  __syncthreads();   // req_flags and the block table visible to the whole block

  const int nb = s_nb;
  // rows per block
  for (int k = warp; k < nb; k += nwarps) {
    const Block bl = s_blk[k];
    int cnt = 0;
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      int n = 0;
      if (b < B && P.req_flags[b] == 0) n = rows_for(bl, P.gamma ? P.gamma[b] : G);
      cnt += __reduce_add_sync(0xffffffffu, n);
    }
    if (lane == 0) s_count[k] = cnt;
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int k = 0; k < nb; ++k) { s_off[k] = acc; acc += s_count[k]; }
    s_off[nb] = acc;
    P.hdr->queue = 0u;
    P.hdr->n_items = (unsigned)acc * (unsigned)P.nch;
    P.hdr->error = 0u;
    P.hdr->n_uncertain = 0u;
  }
  __syncthreads();
  // write the compacted row ids
  for (int k = warp; k < nb; k += nwarps) {
    const Block bl = s_blk[k];
    int off = s_off[k];
    for (int b0 = 0; b0 < B; b0 += 32) {
      const int b = b0 + lane;
      int n = 0, gam = 0;
      if (b < B && P.req_flags[b] == 0) {
        gam = P.gamma ? P.gamma[b] : G;
        n = rows_for(bl, gam);
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
// stats kernel

namespace {

constexpr int F_FIRST = 1, F_LAST = 2, F_TERM = 4;

struct StageDesc {
  int row_id, b, i, kind;
  int chunk, elem0, nvec, flags;
  int head0, nhead, tail0, ntail;
  float c;
  int y;          // draft token whose logit the test needs (-1: none)
  int pad[2];
};

struct EpiSlot {
  int row_id, b, i, kind;
  int chunk, term;
  float xy;       // logit at the draft token if this item held it, else NaN
  int pad;
  Part part[kConsumerWarps];
};

struct __align__(128) StatsSmem {
  unsigned char ring[kStages][kStageBytes];
  uint64_t full[kStages];
  uint64_t empty[kStages];
  uint64_t epi_full[kEpiSlots];
  uint64_t epi_empty[kEpiSlots];
  StageDesc desc[kStages];
  EpiSlot slot[kEpiSlots];
  int abort;
};

__device__ __forceinline__ bool aborted(const StatsSmem& S) {
  return *reinterpret_cast<const volatile int*>(&S.abort) != 0;
}

__device__ __forceinline__ void set_abort(const Params& P, StatsSmem& S) {
  *reinterpret_cast<volatile int*>(&S.abort) = 1;
  atomicOr(&P.hdr->error, (unsigned)SPEC_ST_TIMEOUT);
}

// Bounded wait that also gives up when another role of the CTA aborted.
__device__ __forceinline__ bool wait_bar(StatsSmem& S, uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer();
  while (true) {
    if (mbar_try_wait(bar, parity)) return true;
    if (aborted(S)) return false;
    if (globaltimer() - t0 > kWaitLimitNs) return false;
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

template <int DT, bool ENT>
__device__ __forceinline__ void stage_softmax(RunState& r, const uint4 (&w)[kVecPerThread], float c) {
  using Vec = VecT<DT>;
  constexpr int N = Vec::N;
  const float vm = stage_max<DT, false>(w);
  if (vm > r.m) {
    if (r.m != -INFINITY) {
      const float d = (r.m - vm) * c;
      const float f = ex2(d);
      if (ENT) r.t = f * fmaf(d, r.s, r.t);
      r.s *= f;
    }
    r.m = vm;
    r.mc = vm * c;
  }
  const float mc = r.mc;
  float sv[kVecPerThread], tv[kVecPerThread];
#pragma unroll
  for (int q = 0; q < kVecPerThread; ++q) {
    float x[N], e[N];
    Vec::unpack(w[q], x);
#pragma unroll
    for (int k = 0; k < N; ++k) {
      const float a = fmaf(x[k], c, -mc);
      e[k] = ex2(a);
      if (ENT) x[k] = fmaxf(a, -256.f);       // reuse x for the clamped exponent
    }
    if (N == 8) sv[q] = ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
    else sv[q] = (e[0] + e[1]) + (e[2] + e[3]);
    if (ENT) {
      float t = 0.f;
#pragma unroll
      for (int k = 0; k < N; ++k) t = fmaf(x[k], e[k], t);
      tv[q] = t;
    }
  }
  r.s += (sv[0] + sv[1]) + (sv[2] + sv[3]);
  if (ENT) r.t += (tv[0] + tv[1]) + (tv[2] + tv[3]);
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
__device__ __forceinline__ void run_scalar(RunState& r, float x, int e, float c, bool ent) {
  if (GREEDY) {
    r.nan |= x != x;
    if (x > r.m || (x == r.m && e < r.idx)) { r.m = x; r.idx = e; }
    return;
  }
  if (x > r.m) {
    if (r.m != -INFINITY) {
      const float d = (r.m - x) * c;
      const float f = ex2(d);
      if (ent) r.t = f * fmaf(d, r.s, r.t);
      r.s *= f;
    }
    r.m = x;
    r.mc = x * c;
  }
  const float a = fmaf(x, c, -r.mc);
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

// ---- producer --------------------------------------------------------------

// What the producer needs to stage one claimed item.
struct ItemMeta {
  unsigned q;
  int rid, b, i, kind, chunk, y;
  bool valid, skip;
  float c;
};

template <bool GREEDY>
__device__ __forceinline__ ItemMeta fetch_meta(const Params& P, unsigned q, unsigned n_items) {
  ItemMeta m;
  m.q = q;
  m.valid = q < n_items;
  m.skip = false;
  m.y = -1;
  m.c = 0.f;
  m.rid = m.b = m.i = m.kind = m.chunk = 0;
  if (!m.valid) return m;
  const int nch = P.nch, G = P.G;
  const int slot = (int)(q / (unsigned)nch);
  m.chunk = (int)(q - (unsigned)slot * nch);
  m.rid = __ldg(P.row_list + slot);
  decode_row(m.rid, P.B, G, m.kind, m.b, m.i);
  const int b = m.b, i = m.i;
  // independent loads, issued together
  const int kr = (m.kind == KIND_TARGET || !P.signals_on) ? ld_relaxed(P.known_reject + b) : kNoReject;
  const float T = GREEDY ? 1.f : P.temperature[b];
  const int gam = P.gamma ? P.gamma[b] : G;
  int y = -1;
  // the draft token (sample / one-hot only: signals-only calls have no tokens)
  if (!GREEDY && P.mode != MODE_SIGNALS && i < gam) y = P.draft_tokens[(size_t)b * G + i];
  m.skip = kr < i;             // a reject at an earlier position voids this row
  m.c = GREEDY ? 0.f : scale_of(T);
  m.y = y;
  return m;
}

template <int DT, bool GREEDY>
__device__ void producer_role(const Params& P, StatsSmem& S) {
  constexpr int ES = DT == SPEC_BF16 ? 2 : 4;
  const int G = P.G, V = P.V;
  const int ce = chunk_elems(DT);
  const unsigned n_items = P.hdr->n_items;
  int stage = 0;
  uint32_t phase = 0;
  bool ok = true;
  ItemMeta cur = fetch_meta<GREEDY>(P, atomicAdd(&P.hdr->queue, 1u), n_items);
  while (ok && cur.valid) {
    const unsigned qn = atomicAdd(&P.hdr->queue, 1u);   // next claim, in flight while staging
    if (cur.skip) {
      red_add_release(P.row_arr + cur.rid, 1u + kSkipInc);
    } else {
      const unsigned char* tens = cur.kind == KIND_TARGET ? P.target : P.draft;
      const long long row0 = row_elem_offset(cur.kind, cur.b, cur.i, G, V);
      const int e_begin = cur.chunk * ce;
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
      for (int p = 0; p < npieces; ++p) {
        if (!wait_bar(S, &S.empty[stage], phase ^ 1u)) { ok = false; break; }
        const long long off = (long long)p * kStageBytes;
        const uint32_t bytes = mid > 0 ? (uint32_t)(mid - off < kStageBytes ? mid - off : kStageBytes) : 0u;
        StageDesc& d = S.desc[stage];
        d.row_id = cur.rid; d.b = cur.b; d.i = cur.i; d.kind = cur.kind;
        d.chunk = cur.chunk;
        d.elem0 = (int)((A0 + (uintptr_t)off - rowaddr) / ES);
        d.nvec = (int)(bytes / 16);
        d.flags = (p == 0 ? F_FIRST : 0) | (p == npieces - 1 ? F_LAST : 0);
        d.head0 = e_begin; d.nhead = nhead;
        d.tail0 = e_end - ntail; d.ntail = ntail;
        d.c = cur.c;
        d.y = cur.y;
        if (bytes > 0) {
          mbar_arrive_expect_tx(&S.full[stage], bytes);
          bulk_load(S.ring[stage], reinterpret_cast<const void*>(A0 + (uintptr_t)off), bytes, &S.full[stage]);
        } else {
          mbar_arrive(&S.full[stage]);
        }
        if (++stage == kStages) { stage = 0; phase ^= 1u; }
      }
    }
    cur = fetch_meta<GREEDY>(P, qn, n_items);
  }
  if (ok && wait_bar(S, &S.empty[stage], phase ^ 1u)) {
    S.desc[stage].flags = F_TERM;
    mbar_arrive(&S.full[stage]);
    return;
  }
  // gave up: tell the other roles, then let the copies already in flight land
  set_abort(P, S);
  for (int s = 0; s < kStages; ++s) {
    // the last phase armed on stage s has parity (phase of its last use)
    const uint32_t par = s < stage ? phase : phase ^ 1u;
    const unsigned long long t0 = globaltimer();
    while (!mbar_try_wait(&S.full[s], par) && globaltimer() - t0 < kWaitLimitNs) {
    }
  }
}

// ---- consumers -------------------------------------------------------------

template <int DT, bool GREEDY>
__device__ void consumer_role(const Params& P, StatsSmem& S, int cw, int lane) {
  constexpr int N = VecT<DT>::N;
  const int tid = cw * 32 + lane;
  int stage = 0;
  uint32_t phase = 0;
  int seq = 0;
  RunState r;
  run_reset(r);
  bool ent = false;
  float c = 0.f, xy = __int_as_float(0x7fc00000);
  while (true) {
    if (!wait_bar(S, &S.full[stage], phase)) { set_abort(P, S); return; }
    const StageDesc d = S.desc[stage];
    if (d.flags & F_TERM) {
      // both epilogue warps must see the end: mark two consecutive slots
      for (int e = 0; e < kEpiWarps; ++e) {
        const int es = (seq + e) % kEpiSlots;
        const uint32_t ep = ((uint32_t)((seq + e) / kEpiSlots) & 1u) ^ 1u;
        if (!wait_bar(S, &S.epi_empty[es], ep)) { set_abort(P, S); return; }
        if (tid == 0) S.slot[es].term = 1;
        __syncwarp();
        if (lane == 0) mbar_arrive(&S.epi_full[es]);
      }
      return;
    }
    if (d.flags & F_FIRST) {
      run_reset(r);
      ent = !GREEDY && d.kind == KIND_DRAFT && P.signals_on;
      c = d.c;
      xy = __int_as_float(0x7fc00000);
    }
    const uint4* vec = reinterpret_cast<const uint4*>(S.ring[stage]);
    uint4 w[kVecPerThread];
    load_stage<DT>(vec, d.nvec, tid, w);
    // the logit at the draft token, if this stage holds it (one shared load)
    if (!GREEDY && tid == 0) {
      const int off = d.y - d.elem0;
      if (off >= 0 && off < d.nvec * N) {
        xy = DT == SPEC_BF16 ? __uint_as_float((uint32_t)reinterpret_cast<const unsigned short*>(vec)[off] << 16)
                             : reinterpret_cast<const float*>(vec)[off];
      }
    }
    if (GREEDY) stage_argmax<DT>(r, w, d.elem0, tid);
    else if (ent) stage_softmax<DT, true>(r, w, c);
    else stage_softmax<DT, false>(r, w, c);
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.empty[stage]);
    if (d.flags & F_LAST) {
      if (tid == 0 && (d.nhead > 0 || d.ntail > 0)) {
        const unsigned char* tens = d.kind == KIND_TARGET ? P.target : P.draft;
        const long long row0 = row_elem_offset(d.kind, d.b, d.i, P.G, P.V);
        for (int k = 0; k < d.nhead; ++k) {
          const float x = load_logit(tens, DT, row0 + d.head0 + k);
          if (d.head0 + k == d.y) xy = x;
          run_scalar<GREEDY>(r, x, d.head0 + k, c, ent);
        }
        for (int k = 0; k < d.ntail; ++k) {
          const float x = load_logit(tens, DT, row0 + d.tail0 + k);
          if (d.tail0 + k == d.y) xy = x;
          run_scalar<GREEDY>(r, x, d.tail0 + k, c, ent);
        }
      }
      Part p = to_part(r);
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const Part o = shfl_part(p, off);
        p = GREEDY ? merge_argmax(p, o) : merge_parts(p, o, c, ent);
      }
      const int eslot = seq % kEpiSlots;
      const uint32_t epar = ((uint32_t)(seq / kEpiSlots) & 1u) ^ 1u;
      if (!wait_bar(S, &S.epi_empty[eslot], epar)) { set_abort(P, S); return; }
      if (lane == 0) {
        S.slot[eslot].part[cw] = p;
        if (cw == 0) {
          EpiSlot& E = S.slot[eslot];
          E.row_id = d.row_id; E.b = d.b; E.i = d.i; E.kind = d.kind; E.chunk = d.chunk;
          E.xy = xy;
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.epi_full[eslot]);
      ++seq;
    }
    if (++stage == kStages) { stage = 0; phase ^= 1u; }
  }
}

// ---- epilogue --------------------------------------------------------------

// Acceptance test of position i of request b, both rows complete (tutorial
// page, sections 3.1-3.3).  fp32 on the fp32 row statistics:
//   p(y) = 2^{(x_y - m_p) c} / s_p,  q(y) likewise (1 for one-hot q),
//   accept <=> u q(y) < p(y),  a = min(1, p(y)/q(y)).
// A test closer than 1e-5 (relative) to its threshold is marked and does not
// stop the reading of later rows.
template <bool GREEDY>
__device__ void evaluate_position(const Params& P, int b, int i) {
  const int G = P.G, V = P.V;
  const int tid_t = target_row_id(b, i, G);
  const RowStats tr = ldcg_stats(P.row_stats + tid_t);
  const int y = P.draft_tokens[(size_t)b * G + i];
  int code;
  float a = __int_as_float(0x7fc00000);
  if (GREEDY) {
    if (!row_ok(tr, true)) code = PC_NONFINITE;
    else if (y < 0 || y >= V) code = PC_BAD_TOKEN;
    else code = (y == (tr.idx & ~kIdxNaN)) ? PC_ACCEPT : PC_REJECT;
  } else {
    const bool sample = P.mode == MODE_SAMPLE;
    const int did = draft_row_id(b, i, P.B, G);
    const float u = P.uniforms[(size_t)b * (G + 1) + i];
    const float c = scale_of(P.temperature[b]);
    const float xt = __ldcg(P.row_xy + tid_t);
    RowStats dr{};
    float xd = 0.f;
    if (sample) {
      dr = ldcg_stats(P.row_stats + did);
      xd = __ldcg(P.row_xy + did);
    }
    if (!row_ok(tr, false) || (sample && !row_ok(dr, false))) code = PC_NONFINITE;
    else if (y < 0 || y >= V) code = PC_BAD_TOKEN;
    else if (!(u >= 0.f && u < 1.f)) code = PC_BAD_UNIFORM;
    else {
      const float py = ex2((xt - tr.m) * c) / tr.s;
      const float qy = sample ? ex2((xd - dr.m) * c) / dr.s : 1.f;
      const float uq = u * qy;
      code = uq < py ? PC_ACCEPT : PC_REJECT;
      a = qy > 0.f ? fminf(1.f, py / qy) : (py > 0.f ? 1.f : 0.f);
      if (fabsf(uq - py) <= 1e-5f * fmaxf(uq, py)) {
        code |= PC_UNCERTAIN;
        atomicAdd(&P.hdr->n_uncertain, 1u);
      }
    }
  }
  __stcg(P.pair_res + (size_t)b * (G + 1) + i, code);
  __stcg(P.pair_a + (size_t)b * (G + 1) + i, (double)a);
  if (code != PC_ACCEPT && !(code & PC_UNCERTAIN)) atomicMin(P.known_reject + b, i);
}

// Epilogue warp e handles the items with sequence number = e (mod kEpiWarps).
template <bool GREEDY>
__device__ void epilogue_role(const Params& P, StatsSmem& S, int lane, int e) {
  const int G = P.G, nch = P.nch;
  for (int seq = e;; seq += kEpiWarps) {
    const int eslot = seq % kEpiSlots;
    const uint32_t epar = (uint32_t)(seq / kEpiSlots) & 1u;
    if (!wait_bar(S, &S.epi_full[eslot], epar)) { set_abort(P, S); return; }
    const EpiSlot& E = S.slot[eslot];
    if (E.term) return;
    const int rid = E.row_id, b = E.b, i = E.i, kind = E.kind, chunk = E.chunk;
    const float xy = E.xy;
    Part p = lane < kConsumerWarps ? E.part[lane] : empty_part();
    __syncwarp();
    if (lane == 0) mbar_arrive(&S.epi_empty[eslot]);
    const bool ent = !GREEDY && kind == KIND_DRAFT && P.signals_on;
    const float c = GREEDY ? 0.f : scale_of(P.temperature[b]);
#pragma unroll
    for (int off = 4; off >= 1; off >>= 1) {
      const Part o = shfl_part(p, off);
      p = GREEDY ? merge_argmax(p, o) : merge_parts(p, o, c, ent);
    }
    unsigned old = 0;
    if (lane == 0) {
      stcg_part(P.parts + (size_t)rid * nch + chunk, p);
      if (!(xy != xy)) __stcg(P.row_xy + rid, xy);
      old = atom_add_acqrel(P.row_arr + rid, 1u);   // release: the partial before the count
    }
    old = __shfl_sync(0xffffffffu, old, 0);
    if (((old + 1u) & kCountMask) == (unsigned)nch && (old >> 20) == 0u) {
      // this CTA completed the row: merge its chunks in chunk order
      Part r = empty_part();
      for (int k = lane; k < nch; k += 32) {
        const Part q = ldcg_part(P.parts + (size_t)rid * nch + k);
        r = GREEDY ? merge_argmax(r, q) : merge_parts(r, q, c, ent);
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) {
        const Part o = shfl_part(r, off);
        r = GREEDY ? merge_argmax(r, o) : merge_parts(r, o, c, ent);
      }
      if (lane == 0) {
        stcg_part(reinterpret_cast<Part*>(P.row_stats + rid), r);
        __stcg(P.row_done + rid, 1);
        const int gam = P.gamma ? P.gamma[b] : G;
        int need = 0;
        if (i < gam) {
          if (P.mode == MODE_SAMPLE) need = 2;
          else if ((P.mode == MODE_ONEHOT || P.mode == MODE_GREEDY) && kind == KIND_TARGET) need = 1;
        }
        if (need > 0) {
          // release orders the row stats before the pair arrival
          const unsigned o2 = atom_add_acqrel(P.pair_arr + (size_t)b * (G + 1) + i, 1u);
          if (o2 + 1u == (unsigned)need) evaluate_position<GREEDY>(P, b, i);
        }
      }
    }
  }
}

}  // namespace

template <int DT, bool GREEDY>
__global__ void __launch_bounds__(kStatsThreads, 2) stats_kernel(Params P) {
  extern __shared__ __align__(128) unsigned char smem_raw[];
  StatsSmem& S = *reinterpret_cast<StatsSmem*>(smem_raw);
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
    fence_mbar_init();
  }
  __syncthreads();
  griddep_wait();   // the plan kernel's schedule and counters are ready
  if (warp < kConsumerWarps) consumer_role<DT, GREEDY>(P, S, warp, lane);
  else if (warp == kConsumerWarps) {
    if (lane == 0) producer_role<DT, GREEDY>(P, S);
  } else epilogue_role<GREEDY>(P, S, lane, warp - kConsumerWarps - 1);
  griddep_launch();
}

static size_t stats_smem_bytes() { return sizeof(StatsSmem); }

cudaError_t configure_stats_kernels() {
  const int smem = (int)stats_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(stats_kernel<SPEC_F32, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(stats_kernel<SPEC_F32, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(stats_kernel<SPEC_BF16, false>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e == cudaSuccess)
    e = cudaFuncSetAttribute(stats_kernel<SPEC_BF16, true>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  return e;
}

cudaError_t launch_plan(const Params& P, cudaStream_t s) {
  return launch_ex(plan_kernel, dim3(1), dim3(1024), 0, s, false, P);
}

cudaError_t launch_stats(const Params& P, int grid, cudaStream_t s, bool pdl) {
  const bool greedy = P.mode == MODE_GREEDY;
  void (*k)(Params) = P.dtype == SPEC_BF16 ? (greedy ? stats_kernel<SPEC_BF16, true> : stats_kernel<SPEC_BF16, false>)
                                           : (greedy ? stats_kernel<SPEC_F32, true> : stats_kernel<SPEC_F32, false>);
  return launch_ex(k, dim3(grid), dim3(kStatsThreads), stats_smem_bytes(), s, pdl, P);
}

}  // namespace sv
