// finalize.cu -- per-request decision, final draw and outputs.
//
// Grid (nch2, B) for full-q calls, (1, B) otherwise; 256 threads.  Every CTA
// of request b reads the position results left by stats_kernel and finds the
// first reject k (tutorial page "5.1 投机解码核心原理", section 5.1).  The draw
// that follows (sections 3.2, 3.3, 5.2) is an inverse-CDF search in ascending
// token order, t = u W, token = smallest x with sum_{v<=x} w_v > t:
//   * full-q reject: the weights w = [p_k - q_k]_+ are recomputed from row k of
//     both models; each CTA sums one 4096-token chunk (fp32 terms, fp64 chunk
//     total); the CTA that completes the request locates the chunk where the
//     fp64 prefix crosses t and then the token inside it;
//   * bonus draw (all accepted) and one-hot reject: w is p (without y for
//     one-hot), whose chunk sums are known from the statistics pass; one CTA
//     locates the chunk and rescans only that chunk;
//   * greedy: the token is the argmax kept by the statistics pass.
// Inside the located chunk the token is found by an fp64 walk over fp32
// terms.  The finishing CTA also writes accept_len, tokens, accept_prob, the
// SpecKV signals (H = log2 s - t/s bits, c = 1/s, from the draft rows'
// statistics) and status.
#include <climits>

#include "common.cuh"

namespace sv {
namespace {

enum DrawKind : int { DK_NONE = 0, DK_GREEDY = 1, DK_BONUS = 2, DK_RESIDUAL = 3, DK_ONEHOT = 4 };

struct Decision {
  int status;    // error bits found so far
  int k, gam, kind;
  int draw_row;  // target row id of the draw
};

constexpr int kVoidMask = ~(SPEC_ST_ZERO_RESIDUAL | SPEC_ST_GUARDED);
constexpr double kDrawGuard = 1e-6;   // draws closer than this (relative to W) are counted

// Decision of request b, taken by warp 0 of the CTA: lane i reads what
// position i left (draft row state for the signals, the test result), so all
// loads are issued at once; ballots then find the first reject or error in
// position order.  The result is valid in lane 0.
__device__ Decision decide_warp(const Params& P, int b) {
  Decision D{0, 0, 0, DK_NONE, -1};
  const int G = P.G, lane = threadIdx.x & 31;
  const int flags = P.req_flags[b];
  const int gam = P.gamma ? P.gamma[b] : G;
  const unsigned err = P.hdr->error;
  D.gam = gam;
  if (flags) { D.status = flags; return D; }
  if (err) { D.status = SPEC_ST_TIMEOUT; return D; }
  const bool in = lane < gam;
  // draft rows that feed the signals: all must be complete and finite
  if (P.signals_on) {
    int bad_missing = 0, bad_nonfinite = 0;
    if (in) {
      const int rid = draft_row_id(b, lane, P.B, G);
      const int done = P.row_done[rid];
      const RowStats r = P.row_stats[rid];
      bad_missing = !done;
      bad_nonfinite = done && !row_ok(r, false);
    }
    const unsigned mm = __ballot_sync(0xffffffffu, bad_missing), mn = __ballot_sync(0xffffffffu, bad_nonfinite);
    if (mm | mn) {
      // first bad draft row in order decides which error is reported
      const int f = __ffs(mm | mn) - 1;
      D.status = (mm >> f) & 1u ? SPEC_ST_TIMEOUT : SPEC_ST_NONFINITE;
      return D;
    }
  }
  if (P.mode == MODE_SIGNALS) return D;
  const int code = in ? (P.pair_res[(size_t)b * (G + 1) + lane] & 15) : PC_ACCEPT;
  const unsigned notacc = __ballot_sync(0xffffffffu, code != PC_ACCEPT);
  int k = gam;
  bool rejected = false;
  if (notacc) {
    const int f = __ffs(notacc) - 1;
    const int cf = __shfl_sync(0xffffffffu, code, f);
    if (cf != PC_REJECT) {
      D.status = cf == PC_NONFINITE ? SPEC_ST_NONFINITE
               : cf == PC_BAD_TOKEN ? SPEC_ST_BAD_TOKEN
               : cf == PC_BAD_UNIFORM ? SPEC_ST_BAD_UNIFORM : SPEC_ST_TIMEOUT;
      return D;
    }
    k = f;
    rejected = true;
  }
  D.k = k;
  const int trow = target_row_id(b, k, G);
  const bool greedy = P.mode == MODE_GREEDY;
  if (!rejected) {
    if (!P.row_done[trow]) { D.status = SPEC_ST_TIMEOUT; return D; }
    if (!row_ok(P.row_stats[trow], greedy)) { D.status = SPEC_ST_NONFINITE; return D; }
  }
  D.draw_row = trow;
  if (greedy) { D.kind = DK_GREEDY; return D; }
  const float ud = P.uniforms[(size_t)b * (G + 1) + G];
  if (!(ud >= 0.f && ud < 1.f)) { D.status = SPEC_ST_BAD_UNIFORM; return D; }
  D.kind = !rejected ? DK_BONUS : (P.mode == MODE_SAMPLE ? DK_RESIDUAL : DK_ONEHOT);
  return D;
}

// ---------------------------------------------------------------------------
// block helpers (256 threads)

constexpr int kTile = 4096;              // rescan tile (elements)

struct Scratch {
  double d[kDrawThreads / 32];
  double carry, excl, cprev, cat;
  int found, lastpos, z, last;
  float sig[kDrawThreads];
  float w[kTile + kTile / 16];           // tile weights, one pad word per 16
  float tw[kDrawThreads / 32][8];        // per-warp tile sums
  double tiles[8], tiles_y[8];           // tile sums of a chunk (fp64 totals)
  double h[32], cf[32];
  Decision D;
};

// Sum over the block in a fixed order; every thread gets the total.
__device__ __forceinline__ double block_sum(double v, Scratch& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();
  if (lane == 0) sh.d[warp] = v;
  __syncthreads();
  double tot = 0.0;
#pragma unroll
  for (int w = 0; w < kDrawThreads / 32; ++w) tot += sh.d[w];
  __syncthreads();
  return tot;
}

// Among n non-negative weights get(0..n-1), in order, return the first j
// whose exclusive prefix + weight exceeds t, with that exclusive prefix in
// *excl.  When none does (t >= total, e.g. t = inf), returns the last j with
// a positive weight (*excl = total - its weight) or -1 if all are zero, and
// *total = the sum of all weights (fixed association).
template <class Get>
__device__ int block_locate(int n, Get get, double t, double* excl, Scratch& sh, double* total_out = nullptr) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) { sh.found = INT_MAX; sh.lastpos = -1; sh.carry = 0.0; }
  __syncthreads();
  for (int base = 0; base < n; base += kDrawThreads) {
    const int j = base + threadIdx.x;
    const double v = j < n ? get(j) : 0.0;
    double incl = v;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const double o = __shfl_up_sync(0xffffffffu, incl, d);
      if (lane >= d) incl += o;
    }
    double ex_w = __shfl_up_sync(0xffffffffu, incl, 1);
    if (lane == 0) ex_w = 0.0;
    if (lane == 31) sh.d[warp] = incl;
    __syncthreads();
    double before = sh.carry, tot = sh.carry;
    for (int w = 0; w < kDrawThreads / 32; ++w) {
      if (w < warp) before += sh.d[w];
      tot += sh.d[w];
    }
    const double ex = before + ex_w;
    if (j < n) {
      if (v > 0.0) atomicMax(&sh.lastpos, j);
      if (ex + v > t) atomicMin(&sh.found, j);
    }
    __syncthreads();
    const int f = sh.found;
    if (f != INT_MAX) {
      if (j == f) sh.excl = ex;
      __syncthreads();
      *excl = sh.excl;
      __syncthreads();
      return f;
    }
    if (threadIdx.x == 0) sh.carry = tot;
    __syncthreads();
  }
  const int lp = sh.lastpos;
  const double total = sh.carry;
  __syncthreads();
  if (total_out) *total_out = total;
  if (lp < 0) { *excl = 0.0; return -1; }
  *excl = total - get(lp);
  return lp;
}

// Find the token inside row elements [e0, e1) where the running sum of
// wf(e), started at 0, first exceeds tl.  The range is processed in tiles of
// kTile elements: the block evaluates the tile's weights with coalesced loads
// into shared memory, takes fp32 sums over 16 consecutive elements per thread,
// and an fp64 block scan of those sums (plus the fp64 sum of earlier tiles)
// locates the thread whose range crosses tl; that thread's fp64 walk over its
// 16 weights (continuing into the following ones if rounding requires)
// decides.  Returns the token (every thread) and the fp64 running sums just
// before and after it in *cprev / *cat; when rounding leaves no crossing, the
// last element with positive weight and *cprev = *cat = the full sum.
template <class WF>
__device__ int block_rescan(int e0, int e1, WF wf, double tl, double* cprev, double* cat, Scratch& sh) {
  constexpr int kPer = kTile / kDrawThreads;   // 16
  double base = 0.0;
  if (threadIdx.x == 0) sh.last = -1;
  for (int t0 = e0; t0 < e1; t0 += kTile) {
    const int n = min(kTile, e1 - t0);
    int lastpos = -1;
    for (int i = threadIdx.x; i < kTile; i += kDrawThreads) {
      const float w = i < n ? wf(t0 + i) : 0.f;
      sh.w[i + i / kPer] = w;                          // one pad word per 16: conflict-free rows
      if (w > 0.f) lastpos = t0 + i;
    }
    if (lastpos >= 0) atomicMax(&sh.last, lastpos);
    __syncthreads();
    const float* mine = sh.w + threadIdx.x * (kPer + 1);
    float sum = 0.f;
#pragma unroll
    for (int k = 0; k < kPer; ++k) sum += mine[k];
    sh.sig[threadIdx.x] = sum;
    double ex, tile_total;
    const int js = block_locate(kDrawThreads, [&](int j) { return (double)sh.sig[j]; }, tl - base, &ex, sh,
                                &tile_total);
    // block_locate returns a crossing only when one exists; otherwise the last positive thread
    const bool crossed = js >= 0 && base + ex + (double)sh.sig[js] > tl;
    if (crossed) {
      if ((int)threadIdx.x == js) {
        double C = base + ex, Cp = C;
        int z = -1;
        // walk this thread's weights, then the rest of the tile, in order
        for (int i = js * kPer; i < n; ++i) {
          const float w = sh.w[i + i / kPer];
          Cp = C;
          C += (double)w;
          if (C > tl) { z = t0 + i; break; }
        }
        sh.z = z; sh.cprev = Cp; sh.cat = C;
      }
      __syncthreads();
      if (sh.z >= 0) {
        const int z = sh.z;
        *cprev = sh.cprev;
        *cat = sh.cat;
        __syncthreads();
        return z;
      }
    }
    // no crossing in this tile: carry its total into the next one
    double tot = 0.0;
    {
      double e2;
      block_locate(kDrawThreads, [&](int j) { return (double)sh.sig[j]; }, INFINITY, &e2, sh, &tot);
    }
    base += tot;
    __syncthreads();
  }
  const int z = sh.last;
  *cprev = base;
  *cat = base;
  __syncthreads();
  return z;
}

// Sums of wf over the kTile-element tiles of [e0, e1) (at most 8 tiles):
// every thread takes elements e0 + tid + 256 j (coalesced, all loads in
// flight together), fp32 per thread and tile, fp64 over the block in a fixed
// order.  Results in out[0 .. ntiles-1] (shared), valid after return.
template <class WF>
__device__ int tile_sums(int e0, int e1, WF wf, double* out, Scratch& sh) {
  constexpr int kJ = kTile / kDrawThreads;            // 16 elements per thread and tile
  const int n = e1 - e0;
  const int ntiles = (n + kTile - 1) / kTile;
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  float acc[8];
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    acc[t] = 0.f;
    if (t < ntiles) {
#pragma unroll
      for (int j = 0; j < kJ; ++j) {
        const int i = (int)threadIdx.x + kDrawThreads * (t * kJ + j);
        if (i < n) acc[t] += wf(e0 + i);
      }
    }
  }
#pragma unroll
  for (int t = 0; t < 8; ++t) {
    float v = acc[t];
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
    if (lane == 0) sh.tw[warp][t] = v;
  }
  __syncthreads();
  if (threadIdx.x < 8) {
    double v = 0.0;
    for (int w = 0; w < kDrawThreads / 32; ++w) v += (double)sh.tw[w][threadIdx.x];
    out[threadIdx.x] = v;
  }
  __syncthreads();
  return ntiles;
}

// First tile whose fp64 prefix exceeds tl (in order; else the last positive
// tile), with the prefix before it.  Every thread computes the same answer.
__device__ __forceinline__ int tile_locate(const double* tiles, int ntiles, double tl, double* before) {
  double acc = 0.0;
  int last = -1;
  double last_before = 0.0;
  for (int t = 0; t < ntiles; ++t) {
    if (tiles[t] > 0.0) { last = t; last_before = acc; }
    if (acc + tiles[t] > tl) { *before = acc; return t; }
    acc += tiles[t];
  }
  *before = last_before;
  return last;
}

// ---------------------------------------------------------------------------
// weights

template <int DT>
struct PWeight {           // w = 2^{(x - m)c}, unnormalised p; w(excl) = 0
  const unsigned char* base;
  long long row0;
  float c, mc;
  int excl;
  __device__ float operator()(int e) const {
    if (e == excl) return 0.f;
    return ex2(fmaf(load_logit(base, DT, row0 + e), c, -mc));
  }
};

template <int DT>
struct ResidualWeight {    // w = [p - q]_+
  const unsigned char *tb, *db;
  long long trow0, drow0;
  float c, mpc, mqc, rp, rq;
  __device__ __forceinline__ float term(float xp, float xq) const {
    const float p = ex2(fmaf(xp, c, -mpc)) * rp;
    const float q = ex2(fmaf(xq, c, -mqc)) * rq;
    return fmaxf(p - q, 0.f);
  }
  __device__ float operator()(int e) const {
    return term(load_logit(tb, DT, trow0 + e), load_logit(db, DT, drow0 + e));
  }
};

template <int DT>
__device__ ResidualWeight<DT> residual_weight(const Params& P, int b, int k) {
  const RowStats tr = P.row_stats[target_row_id(b, k, P.G)];
  const RowStats dr = P.row_stats[draft_row_id(b, k, P.B, P.G)];
  ResidualWeight<DT> R;
  R.tb = P.target;
  R.db = P.draft;
  R.trow0 = row_elem_offset(KIND_TARGET, b, k, P.G, P.V);
  R.drow0 = row_elem_offset(KIND_DRAFT, b, k, P.G, P.V);
  R.c = scale_of(P.temperature[b]);
  R.mpc = tr.m * R.c;
  R.mqc = dr.m * R.c;
  R.rp = 1.f / tr.s;
  R.rq = 1.f / dr.s;
  return R;
}

// fp32 sum of the residual over one chunk, strided over the block (fp64 total)
template <int DT>
__device__ double residual_chunk_sum(const ResidualWeight<DT>& R, int e0, int e1, Scratch& sh) {
  constexpr int ES = DT == SPEC_BF16 ? 2 : 4, N = 16 / ES;
  float s = 0.f;
  const uintptr_t at = reinterpret_cast<uintptr_t>(R.tb) + (uintptr_t)((R.trow0 + e0) * ES);
  const uintptr_t ad = reinterpret_cast<uintptr_t>(R.db) + (uintptr_t)((R.drow0 + e0) * ES);
  int body = 0;
  if (((at | ad) & 15u) == 0) {
    body = (e1 - e0) / N;
    const uint4* vt = reinterpret_cast<const uint4*>(at);
    const uint4* vd = reinterpret_cast<const uint4*>(ad);
    for (int v = threadIdx.x; v < body; v += kDrawThreads) {
      const uint4 wt = __ldg(vt + v), wd = __ldg(vd + v);
      if (DT == SPEC_BF16) {
        s += R.term(bf16_lo(wt.x), bf16_lo(wd.x)) + R.term(bf16_hi(wt.x), bf16_hi(wd.x));
        s += R.term(bf16_lo(wt.y), bf16_lo(wd.y)) + R.term(bf16_hi(wt.y), bf16_hi(wd.y));
        s += R.term(bf16_lo(wt.z), bf16_lo(wd.z)) + R.term(bf16_hi(wt.z), bf16_hi(wd.z));
        s += R.term(bf16_lo(wt.w), bf16_lo(wd.w)) + R.term(bf16_hi(wt.w), bf16_hi(wd.w));
      } else {
        s += R.term(__uint_as_float(wt.x), __uint_as_float(wd.x)) + R.term(__uint_as_float(wt.y), __uint_as_float(wd.y));
        s += R.term(__uint_as_float(wt.z), __uint_as_float(wd.z)) + R.term(__uint_as_float(wt.w), __uint_as_float(wd.w));
      }
    }
  }
  for (int e = e0 + body * N + (int)threadIdx.x; e < e1; e += kDrawThreads) s += R(e);
  return block_sum((double)s, sh);
}

// Draw from unnormalised p of target row `rid` (without token excl >= 0).
// Chunk sums come from the statistics pass, except the chunk holding excl,
// which is summed afresh.  Returns the token; sets ZERO_RESIDUAL if the mass
// without excl is zero (then draws from p itself).
template <int DT>
__device__ int draw_from_p(const Params& P, int b, int rid, int excl, float ud, int* st, Scratch& sh,
                           unsigned* n_close) {
  int kind, bb, i;
  decode_row(rid, P.B, P.G, kind, bb, i);
  const RowStats rs = P.row_stats[rid];
  PWeight<DT> W;
  W.base = P.target;
  W.row0 = row_elem_offset(KIND_TARGET, b, i, P.G, P.V);
  W.c = scale_of(P.temperature[b]);
  W.mc = rs.m * W.c;
  W.excl = excl;
  const int ce = chunk_elems(DT);
  const int nch = P.nch;
  const Part* parts = P.parts + (size_t)rid * nch;
  const float c = W.c, m = rs.m;
  auto part_sum = [&](int j) -> double {
    const Part q = parts[j];
    if (!(q.s > 0.f)) return 0.0;
    return (double)(q.s * ex2((q.m - m) * c));
  };
  // the chunk holding the excluded token is summed afresh without it
  int cy = -1, nty = 0;
  double sy = 0.0;
  if (excl >= 0) {
    cy = excl / ce;
    nty = tile_sums(cy * ce, min(cy * ce + ce, P.V), W, sh.tiles_y, sh);
    for (int t = 0; t < nty; ++t) sy += sh.tiles_y[t];
  }
  auto chunk_w = [&](int j) -> double { return j == cy ? sy : part_sum(j); };
  double ex, Wt;
  block_locate(nch, chunk_w, INFINITY, &ex, sh, &Wt);
  if (!(Wt > 0.0)) {
    if (excl < 0) return -1;
    *st |= SPEC_ST_ZERO_RESIDUAL;
    return draw_from_p<DT>(P, b, rid, -1, ud, st, sh, n_close);
  }
  const double t = (double)ud * Wt;
  double excl_pref;
  const int cs = block_locate(nch, chunk_w, t, &excl_pref, sh);
  if (cs < 0) return -1;
  // tiles of the located chunk, then the token inside the located tile
  const int e0 = cs * ce, e1 = min(e0 + ce, P.V);
  const double* tiles = sh.tiles_y;
  int nt = nty;
  if (cs != cy) {
    nt = tile_sums(e0, e1, W, sh.tiles, sh);
    tiles = sh.tiles;
  }
  const double tl = t - excl_pref;
  double tb;
  const int ts = tile_locate(tiles, nt, tl, &tb);
  if (ts < 0) return -1;
  double cp, ca;
  const int z = block_rescan(e0 + ts * kTile, min(e0 + (ts + 1) * kTile, e1), W, tl - tb, &cp, &ca, sh);
  const double tt = tl - tb;
  const double margin = fmin(tt - cp, ca - tt) / Wt;
  if (threadIdx.x == 0 && !(margin >= kDrawGuard)) atomicAdd(n_close, 1u);
  return z;
}

template <int DT>
__device__ int draw_residual(const Params& P, int b, int k, float ud, int* st, Scratch& sh, unsigned* n_close) {
  const int nch2 = P.nch2;
  const double* dp = P.draw_parts + (size_t)b * nch2;
  auto get = [&](int j) -> double { return __ldcg(dp + j); };
  double ex, Wt;
  block_locate(nch2, get, INFINITY, &ex, sh, &Wt);
  if (!(Wt > 0.0)) {
    *st |= SPEC_ST_ZERO_RESIDUAL;
    return draw_from_p<DT>(P, b, target_row_id(b, k, P.G), -1, ud, st, sh, n_close);
  }
  const double t = (double)ud * Wt;
  double excl_pref;
  const int cs = block_locate(nch2, get, t, &excl_pref, sh);
  if (cs < 0) return -1;
  const ResidualWeight<DT> R = residual_weight<DT>(P, b, k);
  double cp, ca;
  const int e0 = cs * kDrawChunkElems, e1 = min(e0 + kDrawChunkElems, P.V);
  const int z = block_rescan(e0, e1, R, t - excl_pref, &cp, &ca, sh);
  const double tl = t - excl_pref;
  const double margin = fmin(tl - cp, ca - tl) / Wt;
  if (threadIdx.x == 0 && !(margin >= kDrawGuard)) atomicAdd(n_close, 1u);
  return z;
}

// ---------------------------------------------------------------------------

template <int DT>
__device__ void finish_request(const Params& P, int b, const Decision& D, Scratch& sh) {
  const int G = P.G;
  int st = D.status;
  int z = -1;
  if (st == 0) {
    const float ud = P.mode == MODE_GREEDY || P.mode == MODE_SIGNALS ? 0.f : P.uniforms[(size_t)b * (G + 1) + G];
    if (D.kind == DK_GREEDY) {
      z = P.row_stats[D.draw_row].idx & ~kIdxNaN;
    } else if (D.kind == DK_BONUS) {
      z = draw_from_p<DT>(P, b, D.draw_row, -1, ud, &st, sh, &P.hdr->n_uncertain);
    } else if (D.kind == DK_ONEHOT) {
      const int y = P.draft_tokens[(size_t)b * G + D.k];
      z = draw_from_p<DT>(P, b, D.draw_row, y, ud, &st, sh, &P.hdr->n_uncertain);
    } else if (D.kind == DK_RESIDUAL) {
      z = draw_residual<DT>(P, b, D.k, ud, &st, sh, &P.hdr->n_uncertain);
    }
    if (D.kind != DK_NONE && z < 0) st |= SPEC_ST_TIMEOUT;   // internal inconsistency: void it
  }
  const bool valid = (st & kVoidMask) == 0;
  const float fnan = __int_as_float(0x7fc00000);
  // signals from the draft rows' statistics
  const bool want_sig = P.signals_on && (P.signals || P.row_signals);
  if (want_sig) {
    const int gam = D.gam;
    if (threadIdx.x < 32) {
      const int i = threadIdx.x;
      double H = 0.0, cf = 0.0;
      if (valid && i < gam) {
        const RowStats r = P.row_stats[draft_row_id(b, i, P.B, G)];
        const double s = (double)r.s;
        H = log2(s) - (double)r.t / s;
        cf = 1.0 / s;
      }
      sh.h[i] = H;
      sh.cf[i] = cf;
      if (P.row_signals && i < G) {
        float* rs = P.row_signals + ((size_t)b * G + i) * 2;
        rs[0] = valid && i < gam ? (float)H : fnan;
        rs[1] = valid && i < gam ? (float)cf : fnan;
      }
    }
    __syncthreads();
    if (threadIdx.x == 0 && P.signals) {
      float* sg = P.signals + (size_t)b * 4;
      if (valid && gam > 0) {
        double hs = 0.0, hm = -INFINITY, cs = 0.0, cm = INFINITY;
        for (int i = 0; i < gam; ++i) {
          hs += sh.h[i]; cs += sh.cf[i];
          hm = fmax(hm, sh.h[i]); cm = fmin(cm, sh.cf[i]);
        }
        sg[0] = (float)(hs / gam); sg[1] = (float)hm; sg[2] = (float)(cs / gam); sg[3] = (float)cm;
      } else {
        sg[0] = sg[1] = sg[2] = sg[3] = fnan;
      }
    }
  }
  if (P.mode != MODE_SIGNALS) {
    const int k = valid ? D.k : 0;
    for (int j = threadIdx.x; j <= G; j += kDrawThreads) {
      int v = -1;
      if (valid) v = j < k ? P.draft_tokens[(size_t)b * G + j] : (j == k ? z : -1);
      P.tokens[(size_t)b * (G + 1) + j] = v;
    }
    if (P.accept_prob)
      for (int j = threadIdx.x; j < G; j += kDrawThreads) {
        float a = fnan;
        if (valid && j < D.gam && j <= D.k) a = (float)P.pair_a[(size_t)b * (G + 1) + j];
        P.accept_prob[(size_t)b * G + j] = a;
      }
    if (threadIdx.x == 0) P.accept_len[b] = k;
  }
  if (threadIdx.x == 0 && P.status) P.status[b] = st;
}

}  // namespace

template <int DT>
__global__ void __launch_bounds__(kDrawThreads) finalize_kernel(Params P) {
  __shared__ Scratch sh;
  griddep_wait();
  const int b = blockIdx.y, chunk = blockIdx.x;
  if (threadIdx.x < 32) {
    const Decision D = decide_warp(P, b);
    if (threadIdx.x == 0) sh.D = D;
  }
  __syncthreads();
  const Decision D = sh.D;
  if (D.status == 0 && D.kind == DK_RESIDUAL) {
    const ResidualWeight<DT> R = residual_weight<DT>(P, b, D.k);
    const int e0 = chunk * kDrawChunkElems, e1 = min(e0 + kDrawChunkElems, P.V);
    const double s = residual_chunk_sum<DT>(R, e0, e1, sh);
    if (threadIdx.x == 0) {
      __stcg(P.draw_parts + (size_t)b * P.nch2 + chunk, s);
      const unsigned old = atom_add_acqrel(P.draw_arr + b, 1u);
      sh.last = (old + 1u == (unsigned)P.nch2);
    }
    __syncthreads();
    if (!sh.last) return;
    __threadfence();
  } else if (chunk != 0) {
    return;
  }
  finish_request<DT>(P, b, D, sh);
}

cudaError_t launch_finalize(const Params& P, dim3 grid, cudaStream_t s, bool pdl) {
  void (*k)(Params) = P.dtype == SPEC_BF16 ? finalize_kernel<SPEC_BF16> : finalize_kernel<SPEC_F32>;
  return launch_ex(k, grid, dim3(kDrawThreads), 0, s, pdl, P);
}

}  // namespace sv
