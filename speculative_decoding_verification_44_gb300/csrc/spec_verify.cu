// spec_verify.cu -- kernels and C ABI of the speculative-decoding verifier
// for GB300 (sm_103a).  Declarations and the contract: include/spec_verify.h.
//
// Launch structure (one launch per call, no host synchronisation):
//   grid = one CTA per (sequence, row slot); slot 0..gamma_max are the target
//   rows, gamma_max+1..2*gamma_max the draft rows.  A CTA whose row the
//   sequence does not use exits at once.  Each used row is analysed by its
//   CTA (sv_row.cuh) and its summary published to the workspace; the CTA that
//   finishes last for a sequence (atomic counter, no waiting) runs the
//   sequence epilogue: the left-to-right acceptance scan, the residual or
//   bonus draw, and the output writes [wrblog §6; rainlin §1].
//
// Sources: [wrblog] "推测解码：草稿模型、接受率、正确性与加速边界" (wrblog.cn);
//          [rainlin] "投机解码" (rainlin-net.pages.dev).
#include "sv_row.cuh"
#include "spec_verify.h"

#include <algorithm>
#include <atomic>
#include <cmath>
#include <cstdint>

namespace sv {

// A sampling rule's domain [wrblog §2.3, §7.2-§7.3]: temperature finite and > 0,
// top_k >= 0, top_p in (0, 1].
__host__ __device__ inline bool rule_ok(const spec_sampling_params_t& p) {
  return isfinite(p.temperature) && p.temperature > 0.0f && p.top_k >= 0 && p.top_p > 0.0f && p.top_p <= 1.0f;
}
// ... and, when the caller promised kept-list rules, 1 <= top_k <= kSmallK (and < V).
__host__ __device__ inline bool rule_ok(const spec_sampling_params_t& p, bool kept_only, int V) {
  return rule_ok(p) && (!kept_only || (p.top_k >= 1 && p.top_k <= kSmallK && p.top_k < V));
}

// A rule prepared for the row kernels (the same arithmetic on host and device).
__host__ __device__ inline RowParams row_params_of(const spec_sampling_params_t& p, int V) {
  RowParams r;
  r.T = p.temperature;
  const double cT = 1.4426950408889634 / static_cast<double>(p.temperature);  // log2(e) / T
  r.cT = static_cast<float>(cT);
  r.cT_lo = static_cast<float>(cT - static_cast<double>(r.cT));
  r.invT = 1.0 / static_cast<double>(p.temperature);
  r.k = (p.top_k >= V) ? 0 : p.top_k;
  r.top_p = p.top_p;
  r.path = (r.k >= 1 && r.k <= kSmallK) ? PATH_STREAM : PATH_FULL;
  int bits = 0;
  for (uint32_t v = static_cast<uint32_t>(V); v; v >>= 1) ++bits;
  const int sh = 62 - bits;
  r.fixed_shift = sh < 24 ? 24 : (sh > 40 ? 40 : sh);
  r.lazy = 0;
  return r;
}

struct ChunkSum;

struct SampleArgs {
  const char* tgt;
  const char* dft;
  const int32_t* tokens;
  const int32_t* gammas;
  const uint8_t* onehot;
  const float* u_acc;
  const float* u_samp;
  RowParams tp, dp;
  const spec_sampling_params_t* tps;   // [B] per-sequence target rules (device), or null
  const spec_sampling_params_t* dps;   // [B] per-sequence draft rules (device), or null
  float beta;           // lenience: beta q stands in for q (1 = the lossless rule)
  int eos;              // end-of-sequence token (-1: none): nothing is committed after it
  int kept_only;        // per-sequence rules promised on the kept-list path
  int B, G, V;
  int aligned;
  size_t row_bytes;
  uint32_t* counters;
  RowStat* stats;
  ListEntry* lists;
  int32_t* out_tokens;
  int32_t* out_nacc;
  float* out_aprob;
  float* out_Z;
  int32_t* out_status;
  int32_t* out_nemit;   // tokens committed, or null
  // full-row draws deferred to draw_kernel (target rows on PATH_FULL)
  int defer;
  int chunk_vecs;       // vectors per draw chunk
  int nchunk;           // chunks per row
  int draw_run;         // chunks per draw CTA (gridDim.y CTAs per sequence)
  uint32_t* dcount;     // [B] chunk CTAs finished (self-cleaning)
  struct DrawRec* drec; // [B]
  // early exit (spec_verify_sample_ex): position-major grid, stop marks
  int early;
  uint32_t* stop_enc;          // [B] G + 1 - (earliest position known to stop), 0 = none (self-cleaning)
  unsigned long long* pairx;   // [B][G] exchange of a position's two draft-token probabilities (self-cleaning)
  ChunkSum* dsum;       // [B][nchunk] weight sums per chunk
  // kept-list kernel: per (sequence, row slot) a block of wpr 16-byte words,
  // a ListRec then the row's kept list in token order
  uint4* fast;
  int wpr;
  int early_logits;     // the caller allows reading logits before the previous grid completes
};

constexpr int kChunkVecs = 4 * kThreads;   // full-row draw: vectors per chunk (four per thread)

// Row record of the kept-list kernel (the first word of a row's block).
struct __align__(16) ListRec {
  float p_tok;      // probability of the draft token this row scores
  int32_t status;   // SEQ_OK, SEQ_NONFINITE or SEQ_EMPTY_SUPPORT
  int32_t n_list;   // kept-list entries that follow
  int32_t pad;
};
static_assert(sizeof(ListRec) == 16 && sizeof(ListEntry) == 16, "kept-list words");

// What draw_kernel needs from the sequence epilogue; j < 0: nothing to draw.
struct DrawRec {
  int32_t j;       // position drawn at (the rejected draft, or gamma for the bonus)
  int32_t flags;   // sequence status flags so far
  int32_t mode;    // ScanCtx mode
  int32_t dj;      // the rejected draft token (mode 3)
};

__device__ __forceinline__ RowStat load_stat(const RowStat* p) {
  RowStat s;
  const uint4* src = reinterpret_cast<const uint4*>(p);
  uint4* d = reinterpret_cast<uint4*>(&s);
  d[0] = __ldcg(src);
  d[1] = __ldcg(src + 1);
  d[2] = __ldcg(src + 2);
  return s;
}
__device__ __forceinline__ ListEntry load_entry(const ListEntry* p) {
  ListEntry e;
  *reinterpret_cast<uint4*>(&e) = __ldcg(reinterpret_cast<const uint4*>(p));
  return e;
}

// Commit nothing [wrblog §15]: all threads of the CTA take part.
__device__ void write_error(const SampleArgs& a, int b, int status) {
  for (int t = threadIdx.x; t <= a.G; t += blockDim.x) a.out_tokens[static_cast<size_t>(b) * (a.G + 1) + t] = -1;
  if (a.out_aprob)
    for (int t = threadIdx.x; t < a.G; t += blockDim.x) a.out_aprob[static_cast<size_t>(b) * a.G + t] = -1.0f;
  if (threadIdx.x == 0) {
    a.out_nacc[b] = -1;
    if (a.out_nemit) a.out_nemit[b] = -1;
    if (a.out_Z) a.out_Z[b] = -1.0f;
    if (a.out_status) a.out_status[b] = status;
    if (a.defer) a.drec[b].j = -1;
  }
}

template <int DT>
__device__ __forceinline__ Row seq_row(const SampleArgs& a, int b, int i, bool draft) {
  const char* base = draft ? a.dft + (static_cast<size_t>(b) * a.G + i) * a.row_bytes
                           : a.tgt + (static_cast<size_t>(b) * (a.G + 1) + i) * a.row_bytes;
  return make_row<DT>(base, a.V, a.aligned != 0);
}

// Probability q(x) of a PATH_STREAM draft row: lookup in its token-sorted list.
__device__ __forceinline__ float list_lookup(const int32_t* tok, const float* p, int n, int x) {
  int lo = 0, hi = n - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    const int t = tok[mid];
    if (t == x) return p[mid];
    if (t < x) lo = mid + 1; else hi = mid - 1;
  }
  return 0.0f;
}

// Z and the inverse-CDF pick over weights held in chunks of 32 entries (entry
// 32c + l is lane l's entry of chunk c, chunk and lane order vocabulary
// order).  wt(c, tok) returns this lane's weight of chunk c and sets its token
// (0 weight past the list's end).  Z is the sum of the chunks' double-float
// scan totals in chunk order; the token is the smallest x with C(x) > u Z, or
// the last entry with weight if rounding leaves none.  Returns -1 (Z_out <= 0)
// when no entry has weight.  Chunk 0 stays in registers, later chunks are
// recomputed (so nothing spills).
template <class WT>
__device__ __forceinline__ int warp_weight_draw(WT wt, int nch, float uf, df& Z_out) {
  const int lane = threadIdx.x & 31;
  int tok0;
  const df w0 = wt(0, tok0);
  const df incl0 = warp_incl_scan_df(w0, lane);
  df Z = df_shfl(incl0, 31);
  for (int c = 1; c < nch; ++c) {
    int tk;
    Z = df_add(Z, df_shfl(warp_incl_scan_df(wt(c, tk), lane), 31));
  }
  Z_out = Z;
  if (!(Z.hi > 0.0f)) return -1;
  const float th = uf * Z.hi;
  const df t = {th, fmaf(uf, Z.hi, -th) + uf * Z.lo};
  df base = df_from(0.0f);
  int last_tok = -1;
  for (int c = 0; c < nch; ++c) {
    int tk = tok0;
    df w = w0, incl = incl0;
    if (c > 0) {
      w = wt(c, tk);
      incl = warp_incl_scan_df(w, lane);
    }
    const bool pos = w.hi > 0.0f;
    const unsigned hit = __ballot_sync(kFull, pos && !df_ge(t, df_add(base, incl)));   // C(x) > u Z
    if (hit) return __shfl_sync(kFull, tk, __ffs(hit) - 1);
    const unsigned any = __ballot_sync(kFull, pos);
    if (any) last_tok = __shfl_sync(kFull, tk, 31 - __clz(any));
    base = df_add(base, df_shfl(incl, 31));
  }
  return last_tok;                                      // rounding left u Z at or above the total
}

// The weight (p - beta q)+ of a kept entry as a double-float [wrblog §5; magicnet
// §8] (beta q is formed exactly, as hi + lo).
__device__ __forceinline__ df residual_weight(const df p, float q, float beta) {
  const float bq = beta * q;
  const df d = df_add(p, {-bq, -fmaf(beta, q, -bq)});
  return d.hi > 0.0f ? d : df_from(0.0f);
}

// Warp-wide inverse-CDF draw over a kept list stored in token order (n <=
// kListCap entries, taken in chunks of 32: entry 32c + l is lane l's entry of
// chunk c, so lane order within a chunk and chunk order are vocabulary order).
// Weights max(0, p - beta q(x)) for a residual [wrblog §5; magicnet §8], p
// itself for the bonus draw; C(x) and Z come from double-float warp scans
// (no float64 arithmetic: that pipe is slow here).  The token is the
// smallest x with C(x) > u Z, or the last entry with weight if rounding
// leaves none.  Z == 0 after a rejection falls back to the draw from p and
// sets SEQ_FLAG_Z_ZERO.  Returns -1 when no entry has weight.
// entry_at(e) gives entry e; q_of(x) gives q(x) (residual draws only).  The
// scan and the pick are warp_weight_draw's.
template <class EntryAt, class QOf>
__device__ __forceinline__ int warp_list_draw(EntryAt entry_at, int n, bool residual, QOf q_of, float beta,
                                              float uf, float& Z_resid, int& flags) {
  const int lane = threadIdx.x & 31;
  const int nch = (n + 31) >> 5;
  for (int pass = 0; pass < 2; ++pass) {
    const bool resid = residual && pass == 0;
    // lane's entry of chunk c: its token and weight (weights (p - beta q)+ when resid)
    const auto weight_of = [&](int c, int& tok) -> df {
      const int e = 32 * c + lane;
      tok = 0x7fffffff;
      if (e >= n) return df_from(0.0f);
      const ListEntry le = entry_at(e);
      tok = le.token;
      const df p = {le.p, le.p_lo};
      return resid ? residual_weight(p, q_of(le.token), beta) : p;
    };
    df Z;
    const int sel = warp_weight_draw(weight_of, nch, uf, Z);
    if (resid) Z_resid = Z.hi;
    if (!(Z.hi > 0.0f)) {
      if (resid) {                                      // Z == 0 after a rejection: draw from p instead
        flags |= SEQ_FLAG_Z_ZERO;
        continue;
      }
      return -1;
    }
    return sel;
  }
  return -1;
}

// q(x) of a kept list in token order: binary search (0 if x is not kept).
__device__ __forceinline__ float kept_q(const ListEntry* ql, int nq, int x) {
  int lo = 0, hi = nq - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    const ListEntry e = ql[mid];
    if (e.token == x) return e.p + e.p_lo;
    if (e.token < x) lo = mid + 1; else hi = mid - 1;
  }
  return 0.0f;
}

// The residual or bonus draw over a PATH_STREAM target row's kept list
// (stored in token order in the workspace), by warp 0 with warp_list_draw.
// The draft's probability comes from its kept list (staged in shared memory
// for the lookups), from its full row, or is the delta of a one-hot draft.
// Block-wide; returns the token to every thread.
template <int DT>
__device__ __noinline__ int list_draw(const SampleArgs& a, int b, int r, bool residual, bool onehot, int dj,
                                      const RowStat& ds, float uf, double& Z_resid, int& flags, Smem& sm) {
  const int tid = threadIdx.x;
  const int slots = 2 * a.G + 1;
  SmemEpi& E = sm.u.e;
  const int nt = E.rs[r].n_list;
  const bool draft_list = residual && !onehot && ds.path == PATH_STREAM;
  const int nq = draft_list ? ds.n_list : 0;
  const ListEntry* tl = a.lists + (static_cast<size_t>(b) * slots + r) * kListCap;
  const ListEntry* ql = a.lists + (static_cast<size_t>(b) * slots + a.G + 1 + r) * kListCap;
  if (tid < nq) {
    const ListEntry q = load_entry(ql + tid);
    E.qtok[tid] = q.token;
    E.qp[tid] = q.p + q.p_lo;
  }
  __syncthreads();
  if (tid < 32) {
    const Row drow = seq_row<DT>(a, b, r, true);
    const auto q_of = [&](int x) -> float {
      if (onehot) return x == dj ? 1.0f : 0.0f;
      if (draft_list) return list_lookup(E.qtok, E.qp, nq, x);
      return full_prob(load_elem<DT>(drow.base, x), static_cast<uint32_t>(x), cut_test(ds.cut), ds.m, ds.cT,
                       ds.invW);
    };
    float Zr = -1.0f;
    const int sel = warp_list_draw([&](int e) { return load_entry(tl + e); }, nt, residual, q_of, a.beta, uf,
                                   Zr, flags);
    if (tid == 0) {
      sm.b_i32[3] = sel;
      if (residual) Z_resid = static_cast<double>(Zr);
    }
  }
  __syncthreads();
  const int sel = sm.b_i32[3];
  __syncthreads();
  return sel;
}

// Per-element weight for the block scan over a PATH_FULL target row.
// mode 0: p; 1: (p - beta q)+ with q a PATH_FULL draft row; 2: (p - beta q)+
// with q a token-sorted list; 3: (p - beta delta_dj)+.
struct ScanCtx {
  Row trow, drow;
  CutTest ctt, ctd;      // kept sets of the target and draft rows
  float mt, md;          // row maxima
  float cTt, cTd, invWt, invWd;
  float beta;            // lenience factor on q
  int mode;
  int dj;
  int nq;
};

template <int DT>
__device__ __forceinline__ int scan_load(const ScanCtx& c, int v, uint4& rt, uint4& rd) {
  const int n = load_vec<DT, false>(c.trow, v, rt);
  rd = make_uint4(0u, 0u, 0u, 0u);
  if (c.mode == 1 && n) load_vec<DT, false>(c.drow, v, rd);
  return n;
}

template <int DT>
__device__ __forceinline__ float scan_weights(const ScanCtx& c, int v, int n, const uint4& rt, const uint4& rd,
                                              const Smem& sm, float (&w)[Elem<DT>::kPer]) {
  constexpr int P = Elem<DT>::kPer;
  float zt[P], zd[P];
  unpack<DT>(rt, zt);
  unpack<DT>(rd, zd);
  float s = 0.0f;
#pragma unroll
  for (int e = 0; e < P; ++e) {
    float we = 0.0f;
    if (e < n) {
      const uint32_t x = static_cast<uint32_t>(v * P + e);
      const float p = full_prob(zt[e], x, c.ctt, c.mt, c.cTt, c.invWt);
      float q = 0.0f;
      if (c.mode == 1) q = full_prob(zd[e], x, c.ctd, c.md, c.cTd, c.invWd);
      else if (c.mode == 2) q = list_lookup(sm.u.e.qtok, sm.u.e.qp, c.nq, static_cast<int>(x));
      else if (c.mode == 3) q = (static_cast<int>(x) == c.dj) ? 1.0f : 0.0f;
      we = c.mode == 0 ? p : fmaxf(p - c.beta * q, 0.0f);
    }
    w[e] = we;
    s += we;
  }
  return s;
}

// Block-wide inverse-CDF draw over a full row in vocabulary order.  Each warp
// owns a contiguous range of vectors, cut into chunks of cv vectors (a
// multiple of 32 x kScanUnroll, at most kScanChunks per warp).  Pass A sums
// the weights per chunk (float per lane, float64 across lanes) with
// kScanUnroll loads in flight per lane; then the chunk holding u Z is found
// from the sums, and one warp re-scans that chunk alone with identical
// arithmetic to locate the first x with C(x) > u Z.
template <int DT>
__device__ __noinline__ int block_scan_draw(ScanCtx c, double u, bool residual, double& Z_resid, int& flags, Smem& sm) {
  constexpr int P = Elem<DT>::kPer;
  constexpr int kStep = 32 * kScanUnroll;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nv = c.trow.nvec;
  const int L = (nv + kWarps - 1) / kWarps;
  const int v0 = warp * L, v1 = min(nv, v0 + L);
  const int per = (L + kScanChunks - 1) / kScanChunks;
  const int cv = max(kStep, (per + kStep - 1) / kStep * kStep);
  const int nch = (L + cv - 1) / cv;
  double (*csum)[kScanChunks] = sm.u.e.csum;
  for (int attempt = 0; attempt < 2; ++attempt) {
    double acc = 0.0;
    for (int k = 0; k < nch; ++k) {
      const int c0 = v0 + k * cv, c1 = min(v1, c0 + cv);
      float ls = 0.0f;
      for (int s = c0; s < c1; s += kStep) {
        uint4 rt[kScanUnroll], rd[kScanUnroll];
        int n[kScanUnroll];
#pragma unroll
        for (int q = 0; q < kScanUnroll; ++q) {
          const int v = s + q * 32 + lane;
          n[q] = v < c1 ? scan_load<DT>(c, v, rt[q], rd[q]) : 0;
        }
#pragma unroll
        for (int q = 0; q < kScanUnroll; ++q) {
          float w[P];
          if (n[q]) ls += scan_weights<DT>(c, s + q * 32 + lane, n[q], rt[q], rd[q], sm, w);
        }
      }
      const double cs = warp_sum_f64(static_cast<double>(ls));
      if (lane == 0) csum[warp][k] = cs;
      acc += cs;
    }
    if (lane == 0) sm.u.e.wtot[warp] = acc;
    __syncthreads();
    if (tid == 0) {
      double Z = 0.0;
      for (int w = 0; w < kWarps; ++w) Z += sm.u.e.wtot[w];
      sm.b_f64[0] = Z;
      // first chunk (warp-major, then chunk) whose range holds t = u Z; the last
      // non-empty chunk if rounding leaves t at or above the total
      const double t = u * Z;
      double start = 0.0, tl = 0.0, last_start = 0.0;
      int W = -1, K = -1, lastW = -1, lastK = -1;
      for (int w = 0; w < kWarps && W < 0; ++w) {
        const int nw = (w * L < nv) ? (min(nv, w * L + L) - w * L + cv - 1) / cv : 0;
        for (int k = 0; k < nw; ++k) {
          const double cs = csum[w][k];
          if (cs > 0.0) {
            lastW = w; lastK = k; last_start = start;
            if (start + cs > t) { W = w; K = k; tl = t - start; break; }
          }
          start += cs;
        }
      }
      if (W < 0) { W = lastW; K = lastK; tl = t - last_start; }
      sm.b_i32[4] = W;
      sm.b_i32[5] = K;
      sm.b_f64[1] = tl;
      sm.b_i32[6] = -1;
    }
    __syncthreads();
    const double Z = sm.b_f64[0];
    if (attempt == 0 && residual) Z_resid = Z;
    if (!(Z > 0.0)) {
      __syncthreads();
      if (attempt == 0 && residual) {     // Z == 0 after a rejection: draw from p instead
        flags |= SEQ_FLAG_Z_ZERO;
        c.mode = 0;
        continue;
      }
      return -1;
    }
    if (warp == sm.b_i32[4]) {
      const double tl = sm.b_f64[1];
      const int c0 = v0 + sm.b_i32[5] * cv, c1 = min(v1, c0 + cv);
      double running = 0.0;
      int last_tok = -1;
      for (int s = c0; s < c1; s += 32) {
        const int v = s + lane;
        float w[P];
        uint4 rt, rd;
        const int n = v < c1 ? scan_load<DT>(c, v, rt, rd) : 0;
        const float ls = n ? scan_weights<DT>(c, v, n, rt, rd, sm, w) : 0.0f;
        if (!n) {
#pragma unroll
          for (int e = 0; e < P; ++e) w[e] = 0.0f;
        }
        const double incl = warp_incl_scan_f64(static_cast<double>(ls), lane);
        const double excl_prev = __shfl_up_sync(kFull, incl, 1);
        const unsigned bal = __ballot_sync(kFull, ls > 0.0f && running + incl > tl);
        // remember the last positive element seen so far (fallback)
        int lp = -1;
#pragma unroll
        for (int e = 0; e < P; ++e) if (w[e] > 0.0f) lp = v * P + e;
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) lp = max(lp, __shfl_xor_sync(kFull, lp, o));
        if (bal) {
          const int Lw = __ffs(bal) - 1;
          if (lane == Lw) {
            const double base = running + (lane > 0 ? excl_prev : 0.0);
            float c32 = 0.0f;
            int tok = -1, lastpos = -1;
#pragma unroll
            for (int e = 0; e < P; ++e) {
              if (w[e] > 0.0f) {
                c32 += w[e];
                lastpos = v * P + e;
                if (tok < 0 && base + static_cast<double>(c32) > tl) tok = v * P + e;
              }
            }
            sm.b_i32[6] = tok >= 0 ? tok : lastpos;
          }
          break;
        }
        if (lp >= 0) last_tok = lp;
        running += __shfl_sync(kFull, incl, 31);
      }
      __syncwarp();
      if (lane == 0 && sm.b_i32[6] < 0) sm.b_i32[6] = last_tok;
    }
    __syncthreads();
    return sm.b_i32[6];
  }
  return -1;
}

// Scan context of a full-row draw at position r.  Block-wide: mode 2 stages
// the draft's kept list, sorted by token, in shared memory.
template <int DT>
__device__ ScanCtx make_scan(const SampleArgs& a, int b, int r, int mode, bool onehot, const RowStat& ts,
                             const RowStat& ds, int dj, Smem& sm) {
  const int tid = threadIdx.x;
  const int slots = 2 * a.G + 1;
  ScanCtx c;
  c.trow = seq_row<DT>(a, b, r, false);
  c.drow = (mode != 0 && !onehot) ? seq_row<DT>(a, b, r, true) : c.trow;
  c.ctt = cut_test(ts.cut);
  c.mt = ts.m;
  c.ctd = cut_test(ds.cut);
  c.md = ds.m;
  c.cTt = ts.cT;
  c.cTd = ds.cT;
  c.invWt = ts.invW;
  c.invWd = ds.invW;
  c.dj = dj;
  c.beta = a.beta;
  c.nq = 0;
  c.mode = mode;
  if (mode == 2) {                 // kept lists are stored in token order
    const ListEntry* ql = a.lists + (static_cast<size_t>(b) * slots + a.G + 1 + r) * kListCap;
    c.nq = ds.n_list;
    if (tid < c.nq) {
      const ListEntry q = load_entry(ql + tid);
      sm.u.e.qtok[tid] = q.token;
      sm.u.e.qp[tid] = q.p + q.p_lo;
    }
    __syncthreads();
  }
  return c;
}

// Sequence epilogue, run by the CTA that analysed the sequence's last row.
template <int DT, bool EX>
__device__ __noinline__ void sample_epilogue(const SampleArgs& a, int b, int gb, bool onehot, Smem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slots = 2 * a.G + 1;
  const RowStat* S = a.stats + static_cast<size_t>(b) * slots;
  const size_t tokb = static_cast<size_t>(b) * a.G;

  // 1. gather, in parallel, every row's status and draft-token probability
  //    (one round trip for the whole CTA; the draft tokens and uniforms were
  //    copied into shared memory while the row streamed)
  SmemEpi& E = sm.u.e;
  for (int t = tid; t < slots; t += kThreads) {
    const bool used = t <= gb || (t > a.G && !onehot && t - a.G - 1 < gb);
    RowStat rs;
    rs.status = SEQ_OK;
    rs.p_tok = 0.0f;
    rs.path = PATH_FULL;
    rs.n_list = 0;
    if (used) rs = load_stat(S + t);
    E.rs[t] = rs;
  }
  if (EX && tid == kThreads - 2) {              // per-sequence rules the sequence uses
    bool ok = true;
    if (a.tps) ok = rule_ok(a.tps[b], a.kept_only != 0, a.V);
    if (a.dps && !onehot) ok = ok && rule_ok(a.dps[b], a.kept_only != 0, a.V);
    sm.b_i32[8] = ok ? 1 : 0;
  }
  __syncthreads();
  // status, in the documented order: tokens, uniforms, rows (lane-parallel, warp 0)
  if (warp == 0) {
    bool bad_tok = false, bad_u = false;
    for (int i = lane; i < gb; i += 32) {
      bad_tok |= sm.seq_tok[i] < 0 || sm.seq_tok[i] >= a.V;
      bad_u |= !(sm.seq_u[i] >= 0.0f && sm.seq_u[i] < 1.0f);
    }
    if (lane == 0) {
      const float us = sm.seq_us;
      bad_u |= !(us >= 0.0f && us < 1.0f);
    }
    int status = SEQ_OK;
    if (__any_sync(kFull, bad_tok)) status = SEQ_BAD_TOKEN;
    else if (__any_sync(kFull, bad_u)) status = SEQ_BAD_UNIFORM;
    else if (EX && !sm.b_i32[8]) status = SEQ_BAD_PARAMS;
    else if (!(EX && a.early)) {
      // rows in order: target 0, draft 0, target 1, draft 1, ..., target gb
      const int norder = 2 * gb + 1;
      for (int base = 0; base < norder && status == SEQ_OK; base += 32) {
        const int o = base + lane;
        int st = SEQ_OK;
        if (o < norder) {
          const int i = o >> 1;
          if ((o & 1) == 0) st = E.rs[i].status;
          else if (!onehot) st = E.rs[a.G + 1 + i].status;
        }
        const unsigned bm = __ballot_sync(kFull, st != SEQ_OK);
        if (bm) status = __shfl_sync(kFull, st, __ffs(bm) - 1);
      }
    }

    // 2. a_i = min(1, p_i(d_i) / q_i(d_i)); accept iff u_i < a_i; stop at the
    //    first rejection -- in the same warp pass, once the status is clean
    int j = gb, flags = 0;
    if (EX && a.early && status == SEQ_OK) {
      // early exit: position by position -- target row i, draft row i, the
      // decision at i -- up to the first failed row or rejected draft; rows
      // after it may not have been read and are ignored
      const auto a_of = [&](int i, bool& zq) {
        const float p = E.rs[i].p_tok;
        const float q = onehot ? 1.0f : E.rs[a.G + 1 + i].p_tok;
        zq = !(q > 0.0f);
        return q > 0.0f ? fminf(1.0f, p / (a.beta * q)) : (p > 0.0f ? 1.0f : 0.0f);
      };
      bool done = false;
      for (int base = 0; base <= gb && !done; base += 32) {
        const int i = base + lane;
        int st = SEQ_OK;
        bool rej = false, zq = false;
        if (i <= gb) {
          st = E.rs[i].status;
          if (st == SEQ_OK && i < gb && !onehot) st = E.rs[a.G + 1 + i].status;
          if (st == SEQ_OK && i < gb) rej = !(sm.seq_u[i] < a_of(i, zq));
        }
        const unsigned ev = __ballot_sync(kFull, i <= gb && (st != SEQ_OK || rej));
        const unsigned zm = __ballot_sync(kFull, zq);
        const int f = ev ? __ffs(ev) - 1 : 31;
        const unsigned upto = (f == 31) ? kFull : ((2u << f) - 1u);
        if (zm & upto) flags |= SEQ_FLAG_ZERO_Q;
        if (ev) {
          const int fst = __shfl_sync(kFull, st, f);
          if (fst != SEQ_OK) status = fst;
          else j = base + f;
          done = true;
        }
      }
      if (status == SEQ_OK && a.out_aprob) {
        for (int i = lane; i < a.G; i += 32) {           // a_i up to the stop, -1 after it
          bool zq;
          a.out_aprob[tokb + i] = (i < gb && i <= j) ? a_of(i, zq) : -1.0f;
        }
      }
    } else if (status == SEQ_OK) {
      for (int base = 0; base < a.G; base += 32) {
        const int i = base + lane;
        bool rej = false, zq = false;
        if (i < gb) {
          const float p = E.rs[i].p_tok;
          const float q = onehot ? 1.0f : E.rs[a.G + 1 + i].p_tok;
          float ai;
          if (q > 0.0f) ai = fminf(1.0f, p / (a.beta * q));   // [magicnet §8]; beta = 1: p / q
          else { ai = p > 0.0f ? 1.0f : 0.0f; zq = true; }
          rej = !(sm.seq_u[i] < ai);
          if (a.out_aprob) a.out_aprob[tokb + i] = ai;
        } else if (i < a.G && a.out_aprob) {
          a.out_aprob[tokb + i] = -1.0f;
        }
        if (j == gb) {
          const unsigned rm = __ballot_sync(kFull, rej);
          const unsigned zm = __ballot_sync(kFull, zq);
          if (rm) {
            const int f = __ffs(rm) - 1;
            j = base + f;
            const unsigned upto = (f == 31) ? kFull : ((2u << f) - 1u);
            if (zm & upto) flags |= SEQ_FLAG_ZERO_Q;
          } else if (zm) {
            flags |= SEQ_FLAG_ZERO_Q;
          }
        }
      }
    }
    // end-of-sequence commit [wrblog §14.3]: the first accepted draft equal to eos ends the block
    int cut = -1;
    if (EX && status == SEQ_OK && a.eos >= 0) {
      for (int base = 0; base < j && cut < 0; base += 32) {
        const unsigned m = __ballot_sync(kFull, base + lane < j && sm.seq_tok[base + lane] == a.eos);
        if (m) cut = base + __ffs(m) - 1;
      }
    }
    if (lane == 0) {
      sm.b_i32[0] = status;
      sm.b_i32[1] = j;
      sm.b_i32[2] = flags;
      sm.b_i32[9] = cut;
    }
  }
  __syncthreads();
  if (sm.b_i32[0] != SEQ_OK) {
    write_error(a, b, sm.b_i32[0]);
    return;
  }
  const int j = sm.b_i32[1];
  int flags = sm.b_i32[2];
  const int cut = EX ? sm.b_i32[9] : -1;
  __syncthreads();
  const size_t ob = static_cast<size_t>(b) * (a.G + 1);
  if (EX && cut >= 0) {
    // an accepted draft is the end-of-sequence token: the committed block ends
    // there, with no replacement or bonus token (so no draw)
    for (int t = tid; t <= a.G; t += kThreads) a.out_tokens[ob + t] = t <= cut ? sm.seq_tok[t] : -1;
    if (tid == 0) {
      a.out_nacc[b] = cut + 1;
      if (a.out_nemit) a.out_nemit[b] = cut + 1;
      if (a.out_Z) a.out_Z[b] = -1.0f;
      if (a.out_status) a.out_status[b] = flags | SEQ_FLAG_EOS;
      if (a.defer) a.drec[b].j = -1;
    }
    return;
  }

  // 3. residual draw at the rejected position, or the bonus draw [wrblog §5, §6]
  const bool residual = j < gb;
  const int r = j;   // == gb when every draft was accepted
  const RowStat ts = E.rs[r];
  RowStat ds;
  ds.path = PATH_FULL; ds.W = 1.0; ds.cut = 0; ds.m = 0.0f; ds.n_list = 0; ds.cT = 0.0f; ds.invW = 1.0f;
  if (residual && !onehot) ds = E.rs[a.G + 1 + r];
  const int dj = residual ? sm.seq_tok[j] : -1;
  const float uf = sm.seq_us;
  double Z_resid = -1.0;
  int tok = -1;
  bool deferred = false;
  if (ts.path == PATH_STREAM) {
    tok = list_draw<DT>(a, b, r, residual, onehot, dj, ds, uf, Z_resid, flags, sm);
    if (a.defer && tid == 0) a.drec[b].j = -1;   // per-sequence rules: nothing for draw_kernel
  } else if (a.defer) {
    // a full-row draw: draw_kernel does it, over runs of chunks, and writes the drawn
    // token, residual_Z and status
    if (tid == 0) {
      DrawRec rec;
      rec.j = j;
      rec.flags = flags;
      rec.mode = !residual ? 0 : (onehot ? 3 : (ds.path == PATH_FULL ? 1 : 2));
      rec.dj = dj;
      a.drec[b] = rec;
    }
    deferred = true;
  } else {
    const int mode = !residual ? 0 : (onehot ? 3 : (ds.path == PATH_FULL ? 1 : 2));
    ScanCtx c = make_scan<DT>(a, b, r, mode, onehot, ts, ds, dj, sm);
    tok = block_scan_draw<DT>(c, static_cast<double>(uf), residual, Z_resid, flags, sm);
  }

  // 4. outputs: accepted drafts, the drawn token, then -1
  for (int t = tid; t <= a.G; t += kThreads) {
    int v = -1;
    if (t < j) v = sm.seq_tok[t];
    else if (t == j) v = tok;
    if (t != j || !deferred) a.out_tokens[ob + t] = v;
  }
  if (tid == 0) {
    a.out_nacc[b] = j;
    if (EX && a.out_nemit) a.out_nemit[b] = j + 1;
    if (!deferred) {
      if (a.out_Z) a.out_Z[b] = residual ? static_cast<float>(Z_resid) : -1.0f;
      if (EX && a.eos >= 0 && tok == a.eos) flags |= SEQ_FLAG_EOS;
      if (a.out_status) a.out_status[b] = flags;
    }
  }
}

// Early exit: the second of position i's two rows to finish (the target row
// alone for a one-hot draft) decides position i exactly as the epilogue will
// -- a_i = min(1, p / (beta q)), rejected iff !(u_i < a_i) -- and marks the
// sequence stopped at i when d_i is rejected or a row of position i failed or
// was not read.  Rows of later positions that start after the mark skip
// their row.  The two rows meet in one 64-bit exchange word per position:
// bit 63 present, bit 62 failed or not read, low 32 bits the row's
// probability of d_i.  Thread 0, after the row summary is final.
__device__ void early_mark(const SampleArgs& a, int b, int i, bool is_draft, bool onehot, bool skipped,
                           const Smem& sm) {
  const RowStat& st = sm.st;
  const bool bad = skipped || st.status != SEQ_OK;
  const unsigned long long mine = (1ull << 63) | (bad ? (1ull << 62) : 0ull) | __float_as_uint(st.p_tok);
  unsigned long long other = (1ull << 63) | __float_as_uint(1.0f);   // one-hot draft: q(d_i) = 1
  if (!onehot) {
    unsigned long long* w = a.pairx + static_cast<size_t>(b) * a.G + i;
    other = atomicExch(w, mine);
    if (other == 0ull) return;        // the other row of position i decides
    *w = 0ull;                        // both rows are in: leave the workspace zero
  }
  bool stop = bad || ((other >> 62) & 1ull);
  if (!stop) {
    const float p = is_draft ? __uint_as_float(static_cast<unsigned>(other)) : st.p_tok;
    const float q = is_draft ? st.p_tok : __uint_as_float(static_cast<unsigned>(other));
    float ai;
    if (q > 0.0f) ai = fminf(1.0f, p / (a.beta * q));
    else ai = p > 0.0f ? 1.0f : 0.0f;
    stop = !(sm.seq_u[i] < ai);
  }
  if (stop) atomicMax(a.stop_enc + b, static_cast<unsigned>(a.G + 1 - i));
}

// EX: the spec_verify_sample_ex features (per-sequence rules, end-of-sequence
// commit, emitted counts, early exit) are compiled in; the plain instantiation
// omits them.
template <int DT, bool EX>
__global__ void __launch_bounds__(kThreads, 5) sample_kernel(const SampleArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  // the full-row draw may be scheduled once every row CTA has started (it
  // waits for this grid to complete before reading anything it wrote)
  grid_launch_dependents();
  const int slots = 2 * a.G + 1;
  int b, slot;
  if (EX && a.early) {
    // position-major: the target and draft rows of position i for every
    // sequence, then position i + 1 (the draft "row" of position G is empty)
    const int i2 = blockIdx.x / (2 * a.B), r2 = blockIdx.x - i2 * 2 * a.B;
    b = r2 >> 1;
    slot = (r2 & 1) ? a.G + 1 + i2 : i2;
  } else {
    b = blockIdx.x / slots;
    slot = blockIdx.x - b * slots;
  }
  const int gb = a.gammas ? a.gammas[b] : a.G;
  const bool onehot = a.dft == nullptr || (a.onehot != nullptr && a.onehot[b] != 0);
  if (gb < 0 || gb > a.G) {
    if (slot == 0) write_error(a, b, SEQ_BAD_LENGTH);
    return;
  }
  const bool is_draft = slot > a.G;
  const int i = is_draft ? slot - a.G - 1 : slot;
  if (!is_draft && i > gb) return;
  if (is_draft && (onehot || i >= gb)) return;

  RowParams P = is_draft ? a.dp : a.tp;
  const spec_sampling_params_t* rules = EX ? (is_draft ? a.dps : a.tps) : nullptr;
  bool rule_valid = true;
  if (EX && rules) {                             // this sequence's own rule [wrblog §15]
    if (threadIdx.x == 0) {
      const spec_sampling_params_t sp = rules[b];
      const bool ok = rule_ok(sp, a.kept_only != 0, a.V);
      sm.b_i32[6] = ok ? 1 : 0;
      if (ok) sm.rowp = row_params_of(sp, a.V);
    }
    __syncthreads();
    rule_valid = sm.b_i32[6] != 0;
    if (rule_valid) P = sm.rowp;
  }
  // A full-row cut that only the full-row draw (which ranks ties itself) and
  // the row's own draft token read may leave open which of its ties of the cut
  // value come first: every target row on that path when draws are deferred,
  // and draft rows whose sequence's target rows take it too (a draft row under
  // a kept-list target is read by the list draw, which needs the exact cut).
  if (a.defer && P.path == PATH_FULL) {
    bool lazy = !is_draft;
    if (is_draft) {
      if (EX && a.tps) {
        if (threadIdx.x == 0) sm.b_i32[5] = row_params_of(a.tps[b], a.V).path;
        __syncthreads();
        lazy = sm.b_i32[5] == PATH_FULL;
      } else {
        lazy = a.tp.path == PATH_FULL;
      }
    }
    P.lazy = lazy ? 1 : 0;
  }
  {
    // the sequence's draft tokens and uniforms, for the epilogue: copied while
    // the row streams, waited for only before this CTA counts its row in
    const size_t tb = static_cast<size_t>(b) * a.G;
    if (static_cast<int>(threadIdx.x) < gb) {
      cp_async4(&sm.seq_tok[threadIdx.x], a.tokens + tb + threadIdx.x);
      cp_async4(&sm.seq_u[threadIdx.x], a.u_acc + tb + threadIdx.x);
    }
    if (threadIdx.x == kThreads - 1) cp_async4(&sm.seq_us, a.u_samp + b);
    cp_async_commit();
  }
  bool skip = false;
  if (EX && a.early && i > 0) {
    // an earlier position of this sequence already stopped it: this row is not read
    if (threadIdx.x == 0) {
      const unsigned se = *reinterpret_cast<volatile const unsigned*>(a.stop_enc + b);
      sm.early_skip = (se != 0u && a.G + 1 - static_cast<int>(se) < i) ? 1 : 0;
    }
    __syncthreads();
    skip = sm.early_skip != 0;
  }
  const Row row = seq_row<DT>(a, b, i, is_draft);
  int dtok = -1;
  if (i < gb) {
    const int t = a.tokens[static_cast<size_t>(b) * a.G + i];
    dtok = (t >= 0 && t < a.V) ? t : -1;
  }
  if (EX && (!rule_valid || skip)) {            // the epilogue reports a bad rule, ignores a skipped row
    if (threadIdx.x == 0) {
      RowStat st;
      st.W = 1.0; st.cut = 0; st.m = 0.0f; st.p_tok = 0.0f; st.status = SEQ_OK; st.n_list = 0;
      st.path = PATH_FULL; st.argmax = -1; st.cT = 0.0f; st.invW = 0.0f;
      sm.st = st;
    }
    __syncthreads();
  } else {
    // early exit: a row of a later position keeps watching its sequence's stop
    // mark and is abandoned if an earlier position stops the sequence meanwhile
    StopCheck sc;
    if (EX && a.early && i > 0) {
      sc.p = a.stop_enc + b;
      sc.thr = static_cast<unsigned>(a.G + 1 - i);
    }
    if (P.path == PATH_STREAM) stream_row<DT>(row, P, dtok, sm, sc);
    else full_row<DT>(row, P, dtok, sm, sc);
  }

  // publish the row summary, then count this row in
  if (threadIdx.x == 0) a.stats[static_cast<size_t>(b) * slots + slot] = sm.st;
  if ((!EX || rule_valid) && P.path == PATH_STREAM) {
    // the kept list, stored in token order (entry e goes to its token's rank)
    static_assert(kListCap <= kThreads, "one thread per kept entry");
    ListEntry* dst = a.lists + (static_cast<size_t>(b) * slots + slot) * kListCap;
    const int n = sm.st.n_list;
    if (threadIdx.x < n) {
      ListEntry le;
      le.p = sm.list_ph[threadIdx.x];
      le.p_lo = sm.list_pl[threadIdx.x];
      le.token = sm.list_tok[threadIdx.x];
      le.pad = 0;
      const int4* lt = reinterpret_cast<const int4*>(sm.list_tok);   // padded with INT_MAX
      int rank = 0;
#pragma unroll 4
      for (int f = 0; f < ((n + 3) >> 2); ++f) {
        const int4 t = lt[f];
        rank += (t.x < le.token ? 1 : 0) + (t.y < le.token ? 1 : 0) + (t.z < le.token ? 1 : 0) +
                (t.w < le.token ? 1 : 0);
      }
      dst[rank] = le;
    }
  }
  cp_async_wait<0>();
  __syncthreads();
  if (threadIdx.x == 0) {
    // release (this CTA's summary and list, ordered before by the barrier) and
    // acquire (the last arriver then sees every other row's) in one atomic
    const unsigned rows_b = static_cast<unsigned>((gb + 1) + (onehot ? 0 : gb));
    if (EX && a.early && i < gb) early_mark(a, b, i, is_draft, onehot, skip, sm);
    const unsigned prev = atom_add_acq_rel_gpu(&a.counters[b], 1u);
    sm.b_i32[7] = (prev + 1u == rows_b) ? 1 : 0;
  }
  __syncthreads();
  if (!sm.b_i32[7]) return;
  sample_epilogue<DT, EX>(a, b, gb, onehot, sm);
  __syncthreads();
  if (threadIdx.x == 0) {                       // leave the workspace reusable
    a.counters[b] = 0u;
    if (EX && a.early) a.stop_enc[b] = 0u;
  }
}

// ------------------------------------------------------------------ kept-list kernel
// The verifier for the common serving case: every used row takes the
// streaming top-k path (1 <= top_k <= kSmallK on both sides, or one-hot
// drafts), rows are 16-byte aligned and gamma_max <= 31.  Each row CTA streams
// its row with the lean loop of lean_stream_row and publishes one contiguous
// block: a ListRec and the kept list in token order.  The CTA that
// finishes last for a sequence reads all of the sequence's blocks in one
// round trip, draws at every position in parallel and lets warp 0 decide:
// status, the left-to-right acceptance scan, the outputs [wrblog §5, §6;
// rainlin §1].  Results are those of sample_kernel: the same row analysis,
// the same acceptance arithmetic and the same draw (warp_list_draw).
constexpr int kGatherWords = static_cast<int>(sizeof(Smem::u)) / 16;   // the epilogue gathers into sm.u

// One position's draw, computed by the epilogue's drawing warps for every
// position while warp 0 decides which one the sequence uses.
struct PosDraw {
  int32_t tok;
  float Z;
  int32_t flags;
  int32_t pad;
};
static_assert(sizeof(PosDraw) * 64 <= sizeof(Smem::sorted), "per-position draws in sm.sorted");

// Sequence epilogue of the kept-list kernel.  `words` (sm.u, dead by now) receives the sequence's row blocks by cp.async, one round
// trip.  Then, at once: warp 0 checks the status and runs the acceptance scan
// (position j of the first rejection, or gamma_b), and warps 1..7 each draw
// for their positions -- the residual draw at i < gamma_b, the bonus draw at
// gamma_b -- since none of the draws depends on j.  Warp 0 then writes the
// outputs with the draw at j.
__device__ __noinline__ void list_epilogue(const SampleArgs& a, int b, int gb, bool onehot, Smem& sm,
                                           uint4* words) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int slots = 2 * a.G + 1, wpr = a.wpr;
  const uint4* src = a.fast + static_cast<size_t>(b) * slots * wpr;
  const int total = slots * wpr;
  for (int t = tid; t < total; t += kThreads) {
    const int s = t / wpr;
    const bool used = s <= gb || (s > a.G && !onehot && s - a.G - 1 < gb);
    if (used) cp_async16(&words[t], src + t);
  }
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  const auto rec = [&](int s) { return *reinterpret_cast<const ListRec*>(&words[s * wpr]); };
  PosDraw* pd = reinterpret_cast<PosDraw*>(sm.sorted);
  const size_t tokb = static_cast<size_t>(b) * a.G;
  const size_t ob = static_cast<size_t>(b) * (a.G + 1);
  if (warp > 0) {
    // the draw at each position i (i < gb: residual weights (p_i - beta q_i)+;
    // i == gb: the bonus draw from p_gb) [wrblog §5, §6; magicnet §8]
    for (int i = warp - 1; i <= gb; i += kWarps - 1) {
      const bool residual = i < gb;
      const int dj = residual ? sm.seq_tok[i] : -1;
      const ListEntry* tl = reinterpret_cast<const ListEntry*>(&words[i * wpr + 1]);
      const ListEntry* ql = reinterpret_cast<const ListEntry*>(&words[(a.G + 1 + i) * wpr + 1]);
      const int nt = min(rec(i).n_list, wpr - 1);
      const int nq = (residual && !onehot) ? min(rec(a.G + 1 + i).n_list, wpr - 1) : 0;
      float Z = -1.0f;
      int flags = 0;
      const int tok = warp_list_draw([&](int e) { return tl[e]; }, nt, residual,
                                     [&](int x) { return onehot ? (x == dj ? 1.0f : 0.0f) : kept_q(ql, nq, x); },
                                     a.beta, sm.seq_us, Z, flags);
      if (lane == 0) {
        PosDraw d;
        d.tok = tok;
        d.Z = Z;
        d.flags = flags;
        d.pad = 0;
        pd[i] = d;
      }
    }
  } else {
    const int i = lane;                         // lane i: position i (gamma_max <= 31)
    // status, in the documented order: tokens, uniforms, rows (target 0, draft 0, target 1, ...)
    bool bad_tok = false, bad_u = false;
    if (i < gb) {
      const int t = sm.seq_tok[i];
      const float u = sm.seq_u[i];
      bad_tok = t < 0 || t >= a.V;
      bad_u = !(u >= 0.0f && u < 1.0f);
    }
    if (lane == 0) bad_u |= !(sm.seq_us >= 0.0f && sm.seq_us < 1.0f);
    int status = SEQ_OK;
    if (__any_sync(kFull, bad_tok)) {
      status = SEQ_BAD_TOKEN;
    } else if (__any_sync(kFull, bad_u)) {
      status = SEQ_BAD_UNIFORM;
    } else {
      int st = SEQ_OK;
      if (i <= gb) {
        st = rec(i).status;
        if (st == SEQ_OK && i < gb && !onehot) st = rec(a.G + 1 + i).status;
      }
      const unsigned bm = __ballot_sync(kFull, st != SEQ_OK);
      if (bm) status = __shfl_sync(kFull, st, __ffs(bm) - 1);
    }
    // a_i = min(1, p_i(d_i) / (beta q_i(d_i))); accept iff u_i < a_i; stop at the first rejection
    int j = gb, flags = 0;
    if (status == SEQ_OK) {
      bool rej = false, zq = false;
      float ai = -1.0f;
      if (i < gb) {
        const float p = rec(i).p_tok;
        const float q = onehot ? 1.0f : rec(a.G + 1 + i).p_tok;
        if (q > 0.0f) ai = fminf(1.0f, p / (a.beta * q));   // [magicnet §8]; beta = 1: p / q
        else { ai = p > 0.0f ? 1.0f : 0.0f; zq = true; }
        rej = !(sm.seq_u[i] < ai);
      }
      if (a.out_aprob && i < a.G) a.out_aprob[tokb + i] = ai;
      const unsigned rm = __ballot_sync(kFull, rej);
      const unsigned zm = __ballot_sync(kFull, zq);
      if (rm) {
        const int f = __ffs(rm) - 1;
        j = f;
        const unsigned upto = (f == 31) ? kFull : ((2u << f) - 1u);
        if (zm & upto) flags |= SEQ_FLAG_ZERO_Q;
      } else if (zm) {
        flags |= SEQ_FLAG_ZERO_Q;
      }
    }
    if (lane == 0) {
      sm.b_i32[0] = status;
      sm.b_i32[1] = j;
      sm.b_i32[2] = flags;
    }
  }
  __syncthreads();
  if (warp != 0) return;
  const int status = sm.b_i32[0], j = sm.b_i32[1];
  const int i = lane;
  if (status != SEQ_OK) {                       // commit nothing [wrblog §15]
    if (i <= a.G) a.out_tokens[ob + i] = -1;
    if (a.out_aprob && i < a.G) a.out_aprob[tokb + i] = -1.0f;
    if (lane == 0) {
      a.out_nacc[b] = -1;
      if (a.out_Z) a.out_Z[b] = -1.0f;
      if (a.out_status) a.out_status[b] = status;
      a.counters[b] = 0u;                       // leave the workspace reusable
    }
    return;
  }
  // outputs: accepted drafts, the drawn token at j, then -1
  const PosDraw d = pd[j];
  if (i <= a.G) a.out_tokens[ob + i] = i < j ? sm.seq_tok[i] : (i == j ? d.tok : -1);
  if (lane == 0) {
    a.out_nacc[b] = j;
    if (a.out_Z) a.out_Z[b] = j < gb ? d.Z : -1.0f;
    if (a.out_status) a.out_status[b] = sm.b_i32[2] | d.flags;
    a.counters[b] = 0u;                         // leave the workspace reusable
  }
}

// A kept-list row's block: its record, then its kept list in token order
// (entry e goes to its token's rank).  Block-wide, after the row analysis.
__device__ __forceinline__ void publish_block(uint4* dst, const Smem& sm) {
  const int tid = threadIdx.x;
  const int n = sm.st.n_list;
  if (tid == 0) {
    ListRec rec;
    rec.p_tok = sm.st.p_tok;
    rec.status = sm.st.status;
    rec.n_list = n;
    rec.pad = 0;
    dst[0] = *reinterpret_cast<const uint4*>(&rec);
  }
  if (tid < n) {
    ListEntry le;
    le.p = sm.list_ph[tid];
    le.p_lo = sm.list_pl[tid];
    le.token = sm.list_tok[tid];
    le.pad = 0;
    const int4* lt = reinterpret_cast<const int4*>(sm.list_tok);   // padded with INT_MAX
    int rank = 0;
#pragma unroll 4
    for (int f = 0; f < ((n + 3) >> 2); ++f) {
      const int4 t = lt[f];
      rank += (t.x < le.token ? 1 : 0) + (t.y < le.token ? 1 : 0) + (t.z < le.token ? 1 : 0) +
              (t.w < le.token ? 1 : 0);
    }
    reinterpret_cast<ListEntry*>(dst + 1)[rank] = le;
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 5) sample_list_kernel(const SampleArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  // Launched as a programmatic dependent: the previous grid in the stream
  // must be complete, its writes visible, before this one reads anything that
  // grid may have written or writes anything itself.  When the caller allows
  // early logits reads (spec_set_early_logits_reads) and there are no
  // per-sequence lengths or one-hot flags, every row is used, so which row a
  // CTA takes needs no memory: it streams its logits first and waits only
  // before reading the draft tokens, so back-to-back calls overlap one call's
  // tail with the next call's stream.  The next call's CTAs may be placed as
  // soon as this grid's CTAs retire.
  const bool stream_first = a.early_logits && a.gammas == nullptr && a.onehot == nullptr;
  if (!stream_first) grid_dependency_wait();
  grid_launch_dependents();
  const int tid = threadIdx.x;
  const int slots = 2 * a.G + 1;
  const int b = blockIdx.x / slots;
  const int slot = blockIdx.x - b * slots;
  const int gb = a.gammas ? a.gammas[b] : a.G;
  const bool onehot = a.dft == nullptr || (a.onehot != nullptr && a.onehot[b] != 0);
  if (gb < 0 || gb > a.G) {
    if (slot == 0) write_error(a, b, SEQ_BAD_LENGTH);
    return;
  }
  const bool is_draft = slot > a.G;
  const int i = is_draft ? slot - a.G - 1 : slot;
  if (!is_draft && i > gb) return;
  if (is_draft && (onehot || i >= gb)) return;
  // the sequence's draft tokens and uniforms, for the epilogue: copied while
  // the row streams (or finishes), waited for only before this CTA counts its row in
  const int32_t* tok = a.tokens + static_cast<size_t>(b) * a.G;
  const float* uacc = a.u_acc + static_cast<size_t>(b) * a.G;
  const float* usamp = a.u_samp + b;
  Smem* smp = &sm;
  auto copy_seq = [=] {
    if (tid < gb) {
      cp_async4(&smp->seq_tok[tid], tok + tid);
      cp_async4(&smp->seq_u[tid], uacc + tid);
    }
    if (tid == kThreads - 1) cp_async4(&smp->seq_us, usamp);
    cp_async_commit();
  };
  if (!stream_first) copy_seq();
  const Row row = seq_row<DT>(a, b, i, is_draft);
  const int V = a.V;
  auto dtok_of = [=] {
    if (stream_first) {
      grid_dependency_wait();
      copy_seq();
    }
    int dtok = -1;
    if (i < gb) {
      const int t = tok[i];
      dtok = (t >= 0 && t < V) ? t : -1;
    }
    return dtok;
  };
  lean_stream_row<DT>(row, is_draft ? a.dp : a.tp, dtok_of, sm);

  publish_block(a.fast + (static_cast<size_t>(b) * slots + slot) * a.wpr, sm);
  cp_async_wait<0>();
  __syncthreads();
  if (tid == 0) {
    // release (this CTA's block, ordered before by the barrier) and acquire
    // (the last arriver then sees every other row's) in one atomic
    const unsigned rows_b = static_cast<unsigned>((gb + 1) + (onehot ? 0 : gb));
    const unsigned prev = atom_add_acq_rel_gpu(&a.counters[b], 1u);
    sm.b_i32[7] = (prev + 1u == rows_b) ? 1 : 0;
  }
  __syncthreads();
  if (!sm.b_i32[7]) return;
  list_epilogue(a, b, gb, onehot, sm, &sm.u.ring[0][0]);
}

// ------------------------------------------------------------------ sampling-mode tree verification
// A draft tree per sequence [baisen §8; magicnet §7]: node 0 is the root, node
// c > 0 carries a token and a parent p_c < c; target row c is the target's
// distribution after the path root..c, draft row c the draft's (the
// distribution the children of c were drawn from).  The children of a node
// are independent proposals from its draft distribution.  Walk from the root
// with the residual r = p_v; try the children in node order with
// min(1, r(x) / q_v(x)); after a rejection r becomes (r - q_v)+ / Z; enter an
// accepted child (r = p_child); when every child is rejected draw from r, at
// a node without children from p_v (the bonus).  With one child per node this
// is the linear verifier (and the arithmetic below is sample_list_kernel's).
//
// Rows take the kept-list path, one CTA per node target row and per node
// draft row (a childless node's draft CTA arrives without reading its row);
// each publishes a block as in sample_list_kernel.  The CTA that finishes last
// for a sequence gathers the row records and the tree, validates, and warp 0
// walks: per visited node one round trip brings the node's target list into
// the lanes (chunks of 32 entries) and its draft list into shared memory.  The
// residual is kept unnormalised, as weights w over the target list's entries
// with S = sum w, so a rejection is w <- (w - S q)+ and S <- sum w without a
// division (S = 1 exactly at a freshly entered node, where w = p).
struct SampleTreeArgs {
  const char* tgt;          // [B][N][V]
  const char* dft;          // [B][N][V]
  const int32_t* tokens;    // [B][N]
  const int32_t* parents;   // [B][N]
  const int32_t* nodes;     // [B] or null (N everywhere)
  const float* u_node;      // [B][N]
  const float* u_samp;      // [B]
  RowParams tp, dp;
  int B, N, V;
  int aligned;
  size_t row_bytes;
  uint32_t* counters;       // [B]
  uint4* blocks;            // [B][2N][wpr]: target rows, then draft rows
  int wpr;
  int32_t* out_tokens;      // [B][N]
  int32_t* out_nacc;        // [B]
  int32_t* out_path;        // [B][N] or null
  float* out_aprob;         // [B][N - 1] or null
  float* out_Z;             // [B] or null
  int32_t* out_status;      // [B] or null
  int early_logits;         // the caller allows reading logits before the previous grid completes
};

// Commit nothing [wrblog §15]: the lanes of one warp.
__device__ void tree_sample_fail(const SampleTreeArgs& a, int b, int status, int lane) {
  const size_t ob = static_cast<size_t>(b) * a.N;
  for (int t = lane; t < a.N; t += 32) {
    a.out_tokens[ob + t] = -1;
    if (a.out_path) a.out_path[ob + t] = -1;
  }
  if (a.out_aprob)
    for (int t = lane; t < a.N - 1; t += 32) a.out_aprob[static_cast<size_t>(b) * (a.N - 1) + t] = -1.0f;
  if (lane == 0) {
    a.out_nacc[b] = -1;
    if (a.out_Z) a.out_Z[b] = -1.0f;
    if (a.out_status) a.out_status[b] = status;
  }
}

// q(x) (hi part) of a kept list in token order: binary search (0 if x is not kept).
__device__ __forceinline__ float kept_q_hi(const ListEntry* ql, int nq, int x) {
  int lo = 0, hi = nq - 1;
  while (lo <= hi) {
    const int mid = (lo + hi) >> 1;
    const int t = ql[mid].token;
    if (t == x) return ql[mid].p;
    if (t < x) lo = mid + 1; else hi = mid - 1;
  }
  return 0.0f;
}

// Sequence epilogue of the tree verifier (max_nodes <= 32: one lane per node);
// kChunks 32-entry chunks cover the longest kept list the rules allow.
template <int kChunks>
__device__ __noinline__ void tree_sample_epilogue(const SampleTreeArgs& a, int b, int n, Smem& sm) {
  const int tid = threadIdx.x, lane = tid & 31;
  const int slots = 2 * a.N, wpr = a.wpr;
  const uint4* blk = a.blocks + static_cast<size_t>(b) * slots * wpr;
  // every row block in one round trip when they fit the gather buffer (the walk
  // then reads shared memory only); otherwise the row records now and each
  // visited node's lists when the walk reaches it
  const bool all = slots * wpr <= kGatherWords;
  uint4* words = &sm.u.ring[0][0];
  const int rstride = all ? wpr : 1;                   // records at words[s * rstride]
  ListEntry* ql = reinterpret_cast<ListEntry*>(&sm.u.ring[0][0] + 64);   // a node's draft list (not all)
  int32_t* tok = sm.seq_tok;
  int32_t* par = sm.list_tok;
  float* un = sm.seq_u;
  const size_t nb = static_cast<size_t>(b) * a.N;
  if (all) {
    for (int t = tid; t < slots * wpr; t += kThreads)
      if ((t / wpr) % a.N < n) cp_async16(&words[t], blk + t);
  } else if (tid < slots && (tid % a.N) < n) {
    cp_async16(&words[tid], blk + static_cast<size_t>(tid) * wpr);
  }
  if (tid < n) {
    cp_async4(&tok[tid], a.tokens + nb + tid);
    cp_async4(&par[tid], a.parents + nb + tid);
    cp_async4(&un[tid], a.u_node + nb + tid);
  }
  if (tid == kThreads - 1) cp_async4(&sm.seq_us, a.u_samp + b);
  cp_async_commit();
  cp_async_wait<0>();
  __syncthreads();
  if (tid >= 32) return;
  const auto rec = [&](int s) { return *reinterpret_cast<const ListRec*>(&words[s * rstride]); };
  // status, in the documented order: node tokens, parents, uniforms, rows in node order
  const int v0 = lane;
  const bool node = v0 >= 1 && v0 < n;
  int status = SEQ_OK;
  if (__any_sync(kFull, node && !(tok[v0] >= 0 && tok[v0] < a.V))) {
    status = SEQ_BAD_TOKEN;
  } else if (__any_sync(kFull, node && !(par[v0] >= 0 && par[v0] < v0))) {
    status = SEQ_BAD_TREE;
  } else if (__any_sync(kFull, (node && !(un[v0] >= 0.0f && un[v0] < 1.0f)) ||
                               (lane == 0 && !(sm.seq_us >= 0.0f && sm.seq_us < 1.0f)))) {
    status = SEQ_BAD_UNIFORM;
  } else {
    int st = SEQ_OK;
    if (v0 < n) {
      st = rec(v0).status;
      if (st == SEQ_OK) st = rec(a.N + v0).status;     // SEQ_OK for a childless node's draft row
    }
    const unsigned bm = __ballot_sync(kFull, st != SEQ_OK);
    if (bm) status = __shfl_sync(kFull, st, __ffs(bm) - 1);
  }
  if (status != SEQ_OK) {
    tree_sample_fail(a, b, status, lane);
    if (lane == 0) a.counters[b] = 0u;
    return;
  }
  const size_t ob = static_cast<size_t>(b) * a.N;
  const size_t ab = static_cast<size_t>(b) * (a.N - 1);
  float a_node = -1.0f;                                 // lane l: a of node l + 1 if it was tried
  int flags = 0;
  int v = 0, L = 0;
  int path_node = lane == 0 ? 0 : -1;                  // lane l: the path's l-th node
  float Z_out = -1.0f;
  int drawn = -1;
  for (;;) {
    const unsigned kids = __ballot_sync(kFull, lane >= 1 && lane < n && par[lane] == v);
    // node v's target list into the lanes, its draft list (if it has children) into shared memory
    const int nt = min(rec(v).n_list, wpr - 1);
    const int nq = kids ? min(rec(a.N + v).n_list, wpr - 1) : 0;
    const int nch = (nt + 31) >> 5;
    const ListEntry* tl = reinterpret_cast<const ListEntry*>((all ? words : blk) + static_cast<size_t>(v) * wpr + 1);
    const ListEntry* gq = reinterpret_cast<const ListEntry*>((all ? words : blk) +
                                                             static_cast<size_t>(a.N + v) * wpr + 1);
    const ListEntry* qv = all ? gq : ql;               // node v's draft list in shared memory
    df w[kChunks];
    int tk[kChunks];
#pragma unroll
    for (int c = 0; c < kChunks; ++c) {
      const int e = 32 * c + lane;
      w[c] = df_from(0.0f);
      tk[c] = 0x7fffffff;
      if (e < nt) {
        const ListEntry le = all ? tl[e] : load_entry(tl + e);
        w[c] = {le.p, le.p_lo};
        tk[c] = le.token;
      }
      if (!all && e < nq) ql[e] = load_entry(gq + e);
    }
    __syncwarp();
    bool unit = true;                                  // w = p and S = 1 exactly
    df S = df_from(1.0f);
    int entered = -1;
    for (unsigned m = kids; m; m &= m - 1) {           // children in node order
      const int c = __ffs(m) - 1;
      const int x = tok[c];
      df px = df_from(0.0f);                           // w(x)
#pragma unroll
      for (int ch = 0; ch < kChunks; ++ch) {
        const unsigned hit = __ballot_sync(kFull, ch < nch && tk[ch] == x);
        if (hit) px = df_shfl(w[ch], __ffs(hit) - 1);
      }
      const float qx = kept_q_hi(qv, nq, x);
      float ac;
      if (qx > 0.0f) {
        ac = unit ? fminf(1.0f, px.hi / (1.0f * qx))   // min(1, p / q), the linear verifier's arithmetic
                  : fminf(1.0f, (px.hi + px.lo) / ((S.hi + S.lo) * qx));
      } else {
        ac = (px.hi > 0.0f) ? 1.0f : 0.0f;
        flags |= SEQ_FLAG_ZERO_Q;
      }
      if (lane == c - 1) a_node = ac;
      if (un[c] < ac) {                                // accept: enter the child
        entered = c;
        break;
      }
      // reject: w <- (w - S q)+ and S <- sum w [wrblog §5]; S == 0 keeps w (R7 of the oracle)
      df nw[kChunks];
#pragma unroll
      for (int ch = 0; ch < kChunks; ++ch) {
        nw[ch] = df_from(0.0f);
        if (ch < nch && 32 * ch + lane < nt) {
          const float q = kept_q(qv, nq, tk[ch]);
          if (unit) {
            nw[ch] = residual_weight(w[ch], q, 1.0f);
          } else {
            const float sq = S.hi * q;                 // S q exactly, as hi + lo
            const df d = df_add(w[ch], {-sq, -(fmaf(S.hi, q, -sq) + S.lo * q)});
            nw[ch] = d.hi > 0.0f ? d : df_from(0.0f);
          }
        }
      }
      df Zn;
      const auto nwt = [&](int ch, int& t) -> df {
        df r = nw[0];
        t = tk[0];
#pragma unroll
        for (int k = 1; k < kChunks; ++k) {
          r = ch == k ? nw[k] : r;
          t = ch == k ? tk[k] : t;
        }
        return r;
      };
      warp_weight_draw(nwt, nch, 0.0f, Zn);            // the total only (the pick is discarded)
      // the residual's mass relative to r = w / S: sum (r - q)+ = Zn / S
      Z_out = unit ? Zn.hi : (Zn.hi + Zn.lo) / (S.hi + S.lo);
      if (Zn.hi > 0.0f) {
#pragma unroll
        for (int ch = 0; ch < kChunks; ++ch) w[ch] = nw[ch];
        S = Zn;
        unit = false;
      } else {
        flags |= SEQ_FLAG_Z_ZERO;
      }
    }
    if (entered >= 0) {
      ++L;
      if (lane == L) path_node = entered;
      v = entered;
      __syncwarp();
      continue;
    }
    // every child rejected: draw from the residual; no children: the bonus from p_v [wrblog §5, §6]
    if (!kids) Z_out = -1.0f;
    const auto wt = [&](int ch, int& t) -> df {
      df r = w[0];
      t = tk[0];
#pragma unroll
      for (int k = 1; k < kChunks; ++k) {
        r = ch == k ? w[k] : r;
        t = ch == k ? tk[k] : t;
      }
      return r;
    };
    df Zd;
    drawn = warp_weight_draw(wt, nch, sm.seq_us, Zd);
    break;
  }
  // outputs: the path's tokens, the drawn token, then -1
  const int pn = __shfl_sync(kFull, path_node, min(lane + 1, 31));   // the path's (lane+1)-th node
  if (lane < a.N) {
    a.out_tokens[ob + lane] = lane < L ? tok[pn] : (lane == L ? drawn : -1);
    if (a.out_path) a.out_path[ob + lane] = lane <= L ? path_node : -1;
  }
  if (a.out_aprob && lane < a.N - 1) a.out_aprob[ab + lane] = a_node;
  if (lane == 0) {
    a.out_nacc[b] = L;
    if (a.out_Z) a.out_Z[b] = Z_out;
    if (a.out_status) a.out_status[b] = flags;
    a.counters[b] = 0u;                                // leave the workspace reusable
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 5) sample_tree_kernel(const SampleTreeArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int tid = threadIdx.x, lane = tid & 31;
  const int slots = 2 * a.N;
  const int b = blockIdx.x / slots;
  const int slot = blockIdx.x - b * slots;
  // with early reads allowed (logits and the tree's parents) and no
  // per-sequence node counts, a row CTA knows from the parents alone whether
  // its row is read, streams it, and waits for the previous grid only before
  // it writes (as in sample_list_kernel)
  const bool stream_first = a.early_logits && a.nodes == nullptr && a.aligned != 0;
  if (!stream_first) grid_dependency_wait();
  grid_launch_dependents();
  const int n = a.nodes ? a.nodes[b] : a.N;
  if (n < 1 || n > a.N) {
    if (slot == 0 && tid < 32) tree_sample_fail(a, b, SEQ_BAD_LENGTH, lane);
    return;
  }
  const bool is_draft = slot >= a.N;
  const int v = is_draft ? slot - a.N : slot;
  if (v >= n) return;
  bool read = true;
  if (is_draft) {                                      // only a node with children has its draft row read
    if (tid < 32) {
      bool has = false;
      for (int c = v + 1 + lane; c < n; c += 32) has |= a.parents[static_cast<size_t>(b) * a.N + c] == v;
      has = __any_sync(kFull, has);
      if (lane == 0) sm.b_i32[6] = has ? 1 : 0;
    }
    __syncthreads();
    read = sm.b_i32[6] != 0;
  }
  uint4* dst = a.blocks + (static_cast<size_t>(b) * slots + slot) * a.wpr;
  if (stream_first && !read) grid_dependency_wait();   // nothing to stream: wait before writing
  if (read) {
    const Row row = make_row<DT>((is_draft ? a.dft : a.tgt) + (static_cast<size_t>(b) * a.N + v) * a.row_bytes,
                                 a.V, a.aligned != 0);
    const RowParams P = is_draft ? a.dp : a.tp;
    if (row.aligned) {
      lean_stream_row<DT>(row, P, [stream_first] {
        if (stream_first) grid_dependency_wait();
        return -1;
      }, sm);
    } else {
      stream_row<DT>(row, P, -1, sm);
    }
    publish_block(dst, sm);
  } else if (tid == 0) {
    ListRec rec;
    rec.p_tok = 0.0f;
    rec.status = SEQ_OK;
    rec.n_list = 0;
    rec.pad = 0;
    dst[0] = *reinterpret_cast<const uint4*>(&rec);
  }
  __syncthreads();
  if (tid == 0) {
    const unsigned prev = atom_add_acq_rel_gpu(&a.counters[b], 1u);
    sm.b_i32[7] = (prev + 1u == static_cast<unsigned>(2 * n)) ? 1 : 0;
  }
  __syncthreads();
  if (!sm.b_i32[7]) return;
  if (a.wpr - 1 <= 32) tree_sample_epilogue<1>(a, b, n, sm);
  else if (a.wpr - 1 <= 64) tree_sample_epilogue<2>(a, b, n, sm);
  else tree_sample_epilogue<kListCap / 32>(a, b, n, sm);
}

// ------------------------------------------------------------------ full-row draw
// The draw at the position the epilogue chose, over whole rows: the inverse
// CDF, in vocabulary order, of w(x) = p(x) (the bonus draw) or
// (p(x) - beta q(x))+ (after a rejection) [wrblog §5, §6].  The rows are cut
// into chunks of kChunkVecs vectors; CTA (b, s) sums the weights of a run of
// draw_run chunks with per-warp partials (no barrier per chunk), and the
// sequence's last CTA finds the chunk holding u Z and the token inside it.
//
// Ties of a cut value.  The streaming sums keep every element whose value is
// at least the row's cut value, ties included, and each chunk also records
// its ties of the target's and of the draft's cut value and how its sum
// changes when the target's, the draft's or both rows' ties are dropped.  A
// row decides its ties either by index (an exact cut: ties up to the index of
// its last kept one) or by rank (a lazy cut, RowStat::n_list = n > 0: the
// first n ties in index order); so a chunk keeps all its ties, none, or --
// the one chunk per row where the last kept tie falls -- some, and that chunk
// is summed again exactly.  No row pass has to locate a lazy cut's last tie,
// and the streaming loop makes no index test.
struct __align__(16) ChunkSum {
  double s;         // weight sum, every tie of either cut value kept
  double d[3];      // change when the target's, the draft's, or both rows' ties are dropped
  int32_t nt, nd;   // ties of the target / draft cut value in the chunk
  int32_t pad[2];
};
static_assert(sizeof(ChunkSum) == 48, "ChunkSum layout");

constexpr int kDrawMaxRun = 32;   // chunks one draw CTA sums (its per-warp partials live in shared memory)
constexpr int kDrawStages = 2;    // half-chunks of each row in flight per draw CTA (bulk copies)
constexpr int kStageVecs = kChunkVecs / 2;
constexpr int kStageRowBytes = kStageVecs * 16;

struct DrawCtx {
  Row trow, drow;
  float kt, kd;            // cut values: kept iff value >= them, ties decided per chunk
  float tt, td;            // tie values (NaN: the row has no cut, nothing ties)
  uint32_t it, id;         // exact cuts: index of the last kept tie
  int nt, nd;              // lazy cuts: ties kept (0: an exact cut)
  float cTt, bt, cTd, bd;  // kept weight 2^(z cT + b), b = -m cT - log2 W: the probability
  float beta;
  int dj, nq;
};

struct DrawPart {
  df s[kDrawMaxRun][kWarps];     // per chunk and warp: weight sum (ties kept)
  df at[kDrawMaxRun][kWarps];    // weight on target ties
  df ad[kDrawMaxRun][kWarps];    // p - w on draft ties
  df ab[kDrawMaxRun][kWarps];    // p - w on elements that tie both cuts
  int nt[kDrawMaxRun][kWarps], nd[kDrawMaxRun][kWarps];
  double xs[2];        // exact sums of the (at most two) chunks where a row's last kept tie falls
  int xk[2];           // their chunk indices (-1: none)
  int xbt[2], xbd[2];  // ties before them (target, draft)
  double tl, Z;        // the draw's offset inside the chosen chunk; the total weight
  int K, Kbt, Kbd;     // the chosen chunk and the ties before it
  DrawCtx ctx;         // the draw's context, for the last CTA's block-wide steps
  RowStat ts;          // the target row's summary (Z = 0 fallback)
  unsigned long long bar[kDrawStages];   // bulk-copy barriers, one per stage
};
// Dynamic shared memory of a draw CTA: Smem, DrawPart, then the stages
// (stage s, row r at kStageRowBytes (2 s + r)).
constexpr size_t kDrawStageOff = (sizeof(Smem) + sizeof(DrawPart) + 127) / 128 * 128;
constexpr size_t kDrawSmem = kDrawStageOff + static_cast<size_t>(kDrawStages) * 2 * kStageRowBytes;
static_assert(static_cast<size_t>(kDrawStages) * 2 * kStageRowBytes >= 32 * kThreads * sizeof(float),
              "the idle stages hold 32 weights per thread for the exact chunk scans");

__device__ __forceinline__ float kept_w(float z, float k, float cT, float b) {
  return z >= k ? fast_exp2(fmaf(z, cT, b)) : 0.0f;
}
template <int MODE>
__device__ __forceinline__ float draw_w(float p, float q, float beta) {
  return MODE == 0 ? p : fmaxf(p - beta * q, 0.0f);
}
// q(x) of the draw, ties kept: 0 (bonus), the draft's full row, its kept list, or one-hot at dj.
template <int MODE>
__device__ __forceinline__ float draw_qk(const DrawCtx& c, float zd, uint32_t x, const Smem& sm) {
  if (MODE == 1) return kept_w(zd, c.kd, c.cTd, c.bd);
  if (MODE == 2) return list_lookup(sm.u.e.qtok, sm.u.e.qp, c.nq, static_cast<int>(x));
  if (MODE == 3) return static_cast<int>(x) == c.dj ? 1.0f : 0.0f;
  return 0.0f;
}

template <int DT, int MODE>
__device__ __forceinline__ int draw_load(const DrawCtx& c, int v, uint4& rt, uint4& rd) {
  const int n = load_vec<DT, false>(c.trow, v, rt);
  rd = make_uint4(0u, 0u, 0u, 0u);
  if (MODE == 1 && n) load_vec<DT, false>(c.drow, v, rd);
  return n;
}

// How a chunk treats one row's ties: 0 keeps them all, 1 none, 2 some.
__device__ __forceinline__ int tie_status(int n, uint32_t idx, uint32_t before, uint32_t cnt, uint32_t x0,
                                          uint32_t x1) {
  if (cnt == 0u) return 0;
  if (n > 0) return before + cnt <= static_cast<uint32_t>(n) ? 0 : (before >= static_cast<uint32_t>(n) ? 1 : 2);
  return x1 - 1u <= idx ? 0 : (x0 > idx ? 1 : 2);
}

// Weights of chunk k with every tie decided: by rank for a lazy cut (bt / bd
// ties before the chunk, then in index order), by index for an exact one.
// The chunk is taken in two halves; in each, thread t takes two consecutive
// vectors, so thread order is index order within a half.  Returns the
// chunk's sum (every thread); with find, also the first token where the
// running sum exceeds tl (else the last token with weight) in *tok.
// Block-wide; c lives in shared memory, and wbuf (shared memory, 32 floats per
// thread) keeps each element's weight for the find.
template <int DT, int MODE>
__device__ __noinline__ double chunk_exact(const DrawCtx& c, int chunk_vecs, int k, int bt, int bd, bool find,
                                           double tl, int* tok, Smem& sm, float* wbuf) {
  constexpr int P = Elem<DT>::kPer;
  constexpr int kVPT = 2;
  static_assert(2 * kVPT * kThreads == kChunkVecs, "two halves of two vectors per thread make a chunk");
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int nv = c.trow.nvec;
  if (tid == 0) { sm.b_i32[5] = -1; sm.b_i32[6] = -1; sm.b_i32[7] = -1; }
  double run = 0.0;            // weight of the halves before
  uint32_t rbt = static_cast<uint32_t>(bt), rbd = static_cast<uint32_t>(bd);
  for (int half = 0; half < 2; ++half) {
    const int v0 = k * chunk_vecs + half * kVPT * kThreads + tid * kVPT;
    uint4 rt[kVPT], rd[kVPT];
    int n[kVPT];
#pragma unroll
    for (int i = 0; i < kVPT; ++i) n[i] = (v0 + i < nv) ? draw_load<DT, MODE>(c, v0 + i, rt[i], rd[i]) : 0;
    uint32_t ct = 0, cd = 0;
#pragma unroll
    for (int i = 0; i < kVPT; ++i) {
      float zt[P], zd[P];
      unpack<DT>(rt[i], zt);
      unpack<DT>(rd[i], zd);
#pragma unroll
      for (int e = 0; e < P; ++e) {
        ct += (e < n[i] && zt[e] == c.tt) ? 1u : 0u;
        cd += (MODE == 1 && e < n[i] && zd[e] == c.td) ? 1u : 0u;
      }
    }
    const uint32_t it_ = warp_incl_scan_u32(ct, lane), id_ = warp_incl_scan_u32(cd, lane);
    if (lane == 31) { sm.nw[warp] = static_cast<int>(it_); sm.red_i[warp] = static_cast<int>(id_); }
    __syncthreads();
    uint32_t rt_ = rbt + it_ - ct, rd_ = rbd + id_ - cd;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) { rt_ += static_cast<uint32_t>(sm.nw[w]); rd_ += static_cast<uint32_t>(sm.red_i[w]); }
      rbt += static_cast<uint32_t>(sm.nw[w]);
      rbd += static_cast<uint32_t>(sm.red_i[w]);
    }
    // the weights, in index order, every tie decided; kept for the find
    float ts = 0.0f;
    int last = -1, e0 = half * kVPT * P;
#pragma unroll
    for (int i = 0; i < kVPT; ++i) {
      float zt[P], zd[P];
      unpack<DT>(rt[i], zt);
      unpack<DT>(rd[i], zd);
#pragma unroll
      for (int e = 0; e < P; ++e) {
        if (e >= n[i]) continue;
        const uint32_t x = static_cast<uint32_t>((v0 + i) * P + e);
        float p = kept_w(zt[e], c.kt, c.cTt, c.bt);
        if (zt[e] == c.tt && !(c.nt > 0 ? rt_++ < static_cast<uint32_t>(c.nt) : x <= c.it)) p = 0.0f;
        float q = draw_qk<MODE>(c, zd[e], x, sm);
        if (MODE == 1 && zd[e] == c.td && !(c.nd > 0 ? rd_++ < static_cast<uint32_t>(c.nd) : x <= c.id)) q = 0.0f;
        const float w = draw_w<MODE>(p, q, c.beta);
        ts += w;
        if (w > 0.0f) last = static_cast<int>(x);
        wbuf[(e0 + i * P + e) * kThreads + tid] = w;
      }
    }
    const df incl = warp_incl_scan_df(df_from(ts), lane);
    if (lane == 31) { sm.red_f[warp] = incl.hi; sm.red_lo[warp] = incl.lo; }
    __syncthreads();
    df base = df_add(incl, df_from(-ts)), tot = df_from(0.0f);
    for (int w = 0; w < kWarps; ++w) {
      const df x = {sm.red_f[w], sm.red_lo[w]};
      if (w < warp) base = df_add(base, x);
      tot = df_add(tot, x);
    }
    const double b0 = run + df_to_double(base);
    if (find && sm.b_i32[5] == -1) {         // not found in an earlier half (same in every thread)
      __syncthreads();
      if (ts > 0.0f && b0 + static_cast<double>(ts) > tl)
        atomicMin(reinterpret_cast<unsigned*>(&sm.b_i32[5]), static_cast<unsigned>(tid));
      if (last >= 0) atomicMax(&sm.b_i32[6], last);
      __syncthreads();
      if (static_cast<unsigned>(sm.b_i32[5]) == static_cast<unsigned>(tid)) {
        float c32 = 0.0f;
        int found = -1;
        for (int i = 0; i < kVPT && found < 0; ++i) {
          for (int e = 0; e < n[i] && found < 0; ++e) {
            const float w = wbuf[(e0 + i * P + e) * kThreads + tid];
            if (w > 0.0f) {
              c32 += w;
              if (b0 + static_cast<double>(c32) > tl) found = (v0 + i) * P + e;
            }
          }
        }
        sm.b_i32[7] = found >= 0 ? found : last;
      }
    }
    run += df_to_double(tot);
    __syncthreads();
  }
  if (find) *tok = sm.b_i32[5] == -1 ? sm.b_i32[6] : sm.b_i32[7];   // rounding: the last weighted token
  __syncthreads();
  return run;
}

template <int DT, int MODE>
__device__ __noinline__ void draw_pick(const SampleArgs& a, int b, int j, int mode, int flags, bool onehot, Smem& sm,
                                       DrawPart& dp, float* wbuf);

// One draw CTA: its run of chunk sums, then (the sequence's last CTA) the draw.
template <int DT, int MODE>
__device__ __noinline__ void draw_body(const SampleArgs& a, int b, const DrawRec rec, const RowStat ts,
                                       const RowStat ds, bool onehot, Smem& sm, DrawPart& dp, uint32_t stage0,
                                       float* wbuf) {
  constexpr int P = Elem<DT>::kPer;
  constexpr int kVPT = 4;
  constexpr int kStep = MODE == 1 ? 2 : 4;   // 64 bytes of each thread in flight per step
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float qnan = __int_as_float(0x7fc00000);
  DrawCtx c;
  c.trow = seq_row<DT>(a, b, rec.j, false);
  c.drow = MODE == 1 ? seq_row<DT>(a, b, rec.j, true) : c.trow;
  const CutTest ctt = cut_test(ts.cut), ctd = cut_test(ds.cut);
  c.kt = ctt.v; c.it = ctt.i;
  c.kd = ctd.v; c.id = ctd.i;
  c.tt = ts.cut != 0ull ? ctt.v : qnan;
  c.td = (MODE == 1 && ds.cut != 0ull) ? ctd.v : qnan;
  c.nt = ts.path == PATH_FULL ? ts.n_list : 0;
  c.nd = (MODE == 1 && ds.path == PATH_FULL) ? ds.n_list : 0;
  c.cTt = ts.cT;
  c.bt = static_cast<float>(-static_cast<double>(ts.m) * static_cast<double>(ts.cT) - log2(ts.W));
  c.cTd = ds.cT;
  c.bd = static_cast<float>(-static_cast<double>(ds.m) * static_cast<double>(ds.cT) - log2(ds.W));
  c.beta = a.beta;
  c.dj = rec.dj;
  c.nq = 0;
  if (MODE == 2) {                 // the draft's kept list, in token order
    const int slots = 2 * a.G + 1;
    const ListEntry* ql = a.lists + (static_cast<size_t>(b) * slots + a.G + 1 + rec.j) * kListCap;
    c.nq = ds.n_list;
    if (tid < c.nq) {
      const ListEntry q = load_entry(ql + tid);
      sm.u.e.qtok[tid] = q.token;
      sm.u.e.qp[tid] = q.p + q.p_lo;
    }
    __syncthreads();
  }
  const int nv = c.trow.nvec;
  const int k0 = blockIdx.y * a.draw_run, k1 = min(a.nchunk, k0 + a.draw_run);

  // 1. this CTA's run of chunks: per-warp partial sums, no barrier per chunk
  float s = 0.0f, at = 0.0f, ad = 0.0f, ab = 0.0f, ct = 0.0f, cd = 0.0f;
  // one element: its weight with ties kept, and the tie bookkeeping
  auto elem = [&](float zt, float zd, uint32_t x) {
    const float pk = kept_w(zt, c.kt, c.cTt, c.bt);
    const float qk = draw_qk<MODE>(c, zd, x, sm);
    const float w = draw_w<MODE>(pk, qk, c.beta);
    s += w;
    const bool tie_t = zt == c.tt;
    at += tie_t ? w : 0.0f;
    ct += tie_t ? 1.0f : 0.0f;
    if (MODE == 1) {
      const bool tie_d = zd == c.td;
      ad += tie_d ? pk - w : 0.0f;
      cd += tie_d ? 1.0f : 0.0f;
      if (tie_t && tie_d) ab += pk - w;
    }
  };
  // a chunk done: this warp's partials
  auto chunk_done = [&](int k) {
    const df ws = warp_sum_df(df_from(s));
    const bool ties = __any_sync(kFull, ct + cd > 0.0f);
    df wt = df_from(0.0f), wd = df_from(0.0f), wb = df_from(0.0f);
    int nt = 0, nd = 0;
    if (ties) {
      wt = warp_sum_df(df_from(at));
      wd = warp_sum_df(df_from(ad));
      wb = warp_sum_df(df_from(ab));
      nt = __reduce_add_sync(kFull, static_cast<unsigned>(ct));
      nd = __reduce_add_sync(kFull, static_cast<unsigned>(cd));
    }
    if (lane == 0) {
      const int r = k - k0;
      dp.s[r][warp] = ws;
      dp.at[r][warp] = wt;
      dp.ad[r][warp] = wd;
      dp.ab[r][warp] = wb;
      dp.nt[r][warp] = nt;
      dp.nd[r][warp] = nd;
    }
    s = at = ad = ab = ct = cd = 0.0f;
  };
  bool stalled = false;
  if (c.trow.aligned && (MODE != 1 || c.drow.aligned)) {
    // bulk copies: one thread streams half-chunks of both rows into the
    // stages, kDrawStages ahead; every thread reads its vectors from there
    // (small stages leave room for three CTAs per SM)
    const uint32_t bar = smem_u32(&dp.bar[0]);
    if (tid == 0) {
      for (int st = 0; st < kDrawStages; ++st) mbar_init(bar + 8u * st, 1u);
      mbar_init_fence();
    }
    __syncthreads();
    const int nq = 2 * (k1 - k0);                   // half-chunks of this CTA's run
    auto issue = [&](int q, int st) {
      const int v0 = (k0 + q / 2) * a.chunk_vecs + (q & 1) * kStageVecs;
      const int nvq = min(kStageVecs, nv - v0);
      const uint32_t bytes = nvq > 0 ? static_cast<uint32_t>(nvq) * 16u : 0u;
      mbar_expect_tx(bar + 8u * st, (MODE == 1 ? 2u : 1u) * bytes);   // 0 bytes: the phase completes now
      if (bytes) {
        bulk_g2s(stage0 + 2u * st * kStageRowBytes, c.trow.base + static_cast<size_t>(v0) * 16, bytes,
                 bar + 8u * st);
        if (MODE == 1)
          bulk_g2s(stage0 + (2u * st + 1u) * kStageRowBytes, c.drow.base + static_cast<size_t>(v0) * 16, bytes,
                   bar + 8u * st);
      }
    };
    if (tid == 0)
      for (int st = 0; st < kDrawStages && st < nq; ++st) issue(st, st);
    int q = 0;
    for (; q < nq; ++q) {
      const int st = q % kDrawStages;
      const bool ok = mbar_wait(bar + 8u * st, static_cast<uint32_t>(q / kDrawStages) & 1u);
      if (__syncthreads_or(!ok)) { stalled = true; break; }
      const int k = k0 + q / 2;
      const int v0 = k * a.chunk_vecs + (q & 1) * kStageVecs, nvq = min(kStageVecs, nv - v0);
      const uint32_t srow = stage0 + 2u * st * kStageRowBytes;
#pragma unroll
      for (int i = 0; i < kStageVecs / kThreads; ++i) {
        const int vl = i * kThreads + tid;
        if (vl >= nvq) continue;
        const uint4 rt = lds128(srow + 16u * vl);
        const uint4 rd = MODE == 1 ? lds128(srow + kStageRowBytes + 16u * vl) : make_uint4(0u, 0u, 0u, 0u);
        float zt[P], zd[P];
        unpack<DT>(rt, zt);
        unpack<DT>(rd, zd);
#pragma unroll
        for (int e = 0; e < P; ++e) elem(zt[e], zd[e], static_cast<uint32_t>((v0 + vl) * P + e));
      }
      if (q & 1) chunk_done(k);
      __syncthreads();                            // every thread is done with stage st
      if (tid == 0 && q + kDrawStages < nq) {
        fence_proxy_async_smem();
        issue(q + kDrawStages, st);
      }
    }
    if (stalled && tid == 0) {
      // let the copies still in flight land (bounded) before the CTA leaves
      for (int r = q; r < min(nq, q + kDrawStages); ++r)
        mbar_wait(bar + 8u * (r % kDrawStages), static_cast<uint32_t>(r / kDrawStages) & 1u);
    }
  } else {
    for (int k = k0; k < k1; ++k) {
      const int v0 = k * a.chunk_vecs;
#pragma unroll 1
      for (int h = 0; h < kVPT; h += kStep) {   // kStep vectors of each row in flight per step
        uint4 rt[kStep], rd[kStep];
        int n[kStep];
#pragma unroll
        for (int i = 0; i < kStep; ++i) {
          const int v = v0 + (h + i) * kThreads + tid;
          n[i] = v < nv ? draw_load<DT, MODE>(c, v, rt[i], rd[i]) : 0;
        }
#pragma unroll
        for (int i = 0; i < kStep; ++i) {
          const int v = v0 + (h + i) * kThreads + tid;
          float zt[P], zd[P];
          unpack<DT>(rt[i], zt);
          unpack<DT>(rd[i], zd);
          if (n[i] == P) {
#pragma unroll
            for (int e = 0; e < P; ++e) elem(zt[e], zd[e], static_cast<uint32_t>(v * P + e));
          } else {
            for (int e = 0; e < n[i]; ++e) elem(zt[e], zd[e], static_cast<uint32_t>(v * P + e));
          }
        }
      }
      chunk_done(k);
    }
  }
  __syncthreads();
  ChunkSum* D = a.dsum + static_cast<size_t>(b) * a.nchunk;
  for (int r = tid; r < k1 - k0; r += kThreads) {
    double sw = 0.0, st = 0.0, sd = 0.0, sb = 0.0;
    int nt = 0, nd = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) {
      sw += df_to_double(dp.s[r][w]);
      st += df_to_double(dp.at[r][w]);
      sd += df_to_double(dp.ad[r][w]);
      sb += df_to_double(dp.ab[r][w]);
      nt += dp.nt[r][w];
      nd += dp.nd[r][w];
    }
    ChunkSum cs;
    cs.s = sw;
    cs.d[0] = -st;             // target ties dropped: their weight goes
    cs.d[1] = sd;              // draft ties dropped: their weight becomes p
    cs.d[2] = sd - st - sb;    // both: target ties lose their weight, draft-only ties become p
    cs.nt = stalled ? 0 : nt;
    cs.nd = stalled ? 0 : nd;
    cs.pad[0] = stalled ? 1 : 0;   // this CTA's copies stalled: the sequence reports SEQ_STALLED
    cs.pad[1] = 0;
    D[k0 + r] = cs;
  }
  __syncthreads();
  if (tid == 0) {
    // release this CTA's chunk sums, acquire the others' (the last arriver reads them all)
    const unsigned prev = atom_add_acq_rel_gpu(&a.dcount[b], 1u);
    sm.b_i32[7] = (prev + 1u == gridDim.y) ? 1 : 0;
  }
  __syncthreads();
  if (!sm.b_i32[7]) return;
  if (tid == 0) {
    dp.ctx = c;
    dp.ts = ts;
  }
  __syncthreads();
  // the stages are idle now (every copy was consumed): they hold the exact
  // scans' per-element weights
  draw_pick<DT, MODE>(a, b, rec.j, rec.mode, rec.flags, onehot, sm, dp, wbuf);
}

// The sequence's last draw CTA: each chunk's tie statuses, exact sums where a
// row's last kept tie falls, Z, the chunk holding u Z and the token inside
// it; then the outputs.
template <int DT, int MODE>
__device__ __noinline__ void draw_pick(const SampleArgs& a, int b, int j, int mode, int flags, bool onehot, Smem& sm,
                                       DrawPart& dp, float* wbuf) {
  constexpr int P = Elem<DT>::kPer;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const DrawCtx& c = dp.ctx;
  const ChunkSum* D = a.dsum + static_cast<size_t>(b) * a.nchunk;
  const double u = static_cast<double>(a.u_samp[b]);
  const uint32_t cx = static_cast<uint32_t>(a.chunk_vecs) * P;   // elements per chunk
  // chunk k's weight under the ties it keeps; -1: some of a row's ties (summed exactly)
  auto chunk_w = [&](int k, const ChunkSum& cs, uint32_t bt, uint32_t bd) -> double {
    const uint32_t x0 = static_cast<uint32_t>(k) * cx, x1 = min(static_cast<uint32_t>(a.V), x0 + cx);
    const int st = tie_status(c.nt, c.it, bt, static_cast<uint32_t>(cs.nt), x0, x1);
    const int sd = tie_status(c.nd, c.id, bd, static_cast<uint32_t>(cs.nd), x0, x1);
    if (st == 2 || sd == 2) return -1.0;
    return fmax(cs.s + (st ? (sd ? cs.d[2] : cs.d[0]) : (sd ? cs.d[1] : 0.0)), 0.0);
  };
  auto load_cs = [&](int k) {
    ChunkSum cs;
    cs.s = 0.0; cs.d[0] = cs.d[1] = cs.d[2] = 0.0; cs.nt = cs.nd = 0; cs.pad[0] = cs.pad[1] = 0;
    if (k < a.nchunk) {
      cs.s = __ldcg(&D[k].s);
      cs.d[0] = __ldcg(&D[k].d[0]);
      cs.d[1] = __ldcg(&D[k].d[1]);
      cs.d[2] = __ldcg(&D[k].d[2]);
      cs.nt = __ldcg(&D[k].nt);
      cs.nd = __ldcg(&D[k].nd);
      cs.pad[0] = __ldcg(&D[k].pad[0]);
    }
    return cs;
  };
  if (warp == 0) {
    if (lane == 0) { dp.xk[0] = dp.xk[1] = -1; dp.K = 0; }
    __syncwarp();
    uint32_t bt = 0, bd = 0;
    int nx = 0;
    bool stalled = false;
    for (int base = 0; base < a.nchunk; base += 32) {
      const int k = base + lane;
      const ChunkSum cs = load_cs(k);
      stalled = __any_sync(kFull, cs.pad[0] != 0) || stalled;
      const uint32_t it_ = warp_incl_scan_u32(static_cast<uint32_t>(cs.nt), lane);
      const uint32_t id_ = warp_incl_scan_u32(static_cast<uint32_t>(cs.nd), lane);
      const uint32_t kbt = bt + it_ - cs.nt, kbd = bd + id_ - cs.nd;
      const bool exact = k < a.nchunk && chunk_w(k, cs, kbt, kbd) < 0.0;
      const unsigned m = __ballot_sync(kFull, exact);
      if (exact) {
        const int slot = nx + __popc(m & ((1u << lane) - 1u));
        if (slot < 2) { dp.xk[slot] = k; dp.xbt[slot] = static_cast<int>(kbt); dp.xbd[slot] = static_cast<int>(kbd); }
      }
      nx += __popc(m);
      bt += __shfl_sync(kFull, it_, 31);
      bd += __shfl_sync(kFull, id_, 31);
    }
    if (lane == 0 && stalled) dp.K = -2;
  }
  __syncthreads();
  if (dp.K == -2) {                     // a CTA of this draw stalled: commit nothing
    const size_t ob = static_cast<size_t>(b) * (a.G + 1);
    for (int t = tid; t <= a.G; t += kThreads) a.out_tokens[ob + t] = -1;
    if (tid == 0) {
      a.out_nacc[b] = -1;
      if (a.out_nemit) a.out_nemit[b] = -1;
      if (a.out_Z) a.out_Z[b] = -1.0f;
      if (a.out_status) a.out_status[b] = SEQ_STALLED;
      a.dcount[b] = 0u;
    }
    return;
  }
  for (int x = 0; x < 2; ++x) {
    if (dp.xk[x] < 0) continue;
    const double v = chunk_exact<DT, MODE>(c, a.chunk_vecs, dp.xk[x], dp.xbt[x], dp.xbd[x], false, 0.0, nullptr, sm,
                                           wbuf);
    if (tid == 0) dp.xs[x] = fmax(v, 0.0);
  }
  __syncthreads();
  if (warp == 0) {
    // Z, then the first chunk (with weight) whose range holds t = u Z; the
    // last chunk with weight if rounding leaves t at or above the total
    double Z = 0.0;
    for (int pass = 0; pass < 2; ++pass) {
      const double t = u * Z;
      uint32_t bt = 0, bd = 0;
      double run = 0.0, tl = 0.0, last_start = 0.0, tot = 0.0;
      int K = -1, lastK = -1, Kbt = 0, Kbd = 0, lbt = 0, lbd = 0;
      for (int base = 0; base < a.nchunk; base += 32) {
        const int k = base + lane;
        const ChunkSum cs = load_cs(k);
        const uint32_t it_ = warp_incl_scan_u32(static_cast<uint32_t>(cs.nt), lane);
        const uint32_t id_ = warp_incl_scan_u32(static_cast<uint32_t>(cs.nd), lane);
        const uint32_t kbt = bt + it_ - cs.nt, kbd = bd + id_ - cs.nd;
        double w = 0.0;
        if (k < a.nchunk) {
          w = chunk_w(k, cs, kbt, kbd);
          if (w < 0.0) w = (k == dp.xk[0]) ? dp.xs[0] : dp.xs[1];
        }
        bt += __shfl_sync(kFull, it_, 31);
        bd += __shfl_sync(kFull, id_, 31);
        if (pass == 0) {
          tot += warp_sum_f64(w);
          continue;
        }
        if (K >= 0) continue;
        const double incl = warp_incl_scan_f64(w, lane);
        const unsigned hit = __ballot_sync(kFull, w > 0.0 && run + incl > t);
        const unsigned pos = __ballot_sync(kFull, w > 0.0);
        if (hit) {
          const int L = __ffs(hit) - 1;
          K = base + L;
          tl = t - (run + __shfl_sync(kFull, incl - w, L));
          Kbt = static_cast<int>(__shfl_sync(kFull, kbt, L));
          Kbd = static_cast<int>(__shfl_sync(kFull, kbd, L));
        } else if (pos) {
          const int L = 31 - __clz(pos);
          lastK = base + L;
          last_start = run + __shfl_sync(kFull, incl - w, L);
          lbt = static_cast<int>(__shfl_sync(kFull, kbt, L));
          lbd = static_cast<int>(__shfl_sync(kFull, kbd, L));
        }
        run += __shfl_sync(kFull, incl, 31);
      }
      if (pass == 0) {
        Z = tot;
        continue;
      }
      if (K < 0) { K = lastK; tl = t - last_start; Kbt = lbt; Kbd = lbd; }
      if (lane == 0) { dp.Z = Z; dp.tl = tl; dp.K = K; dp.Kbt = Kbt; dp.Kbd = Kbd; }
    }
  }
  __syncthreads();
  const double Z = dp.Z;
  int tok = -1;
  if (!(Z > 0.0) || dp.K < 0) {
    // no weight at all: after a rejection, draw from p over the whole row
    if (mode != 0) {
      flags |= SEQ_FLAG_Z_ZERO;
      RowStat t2 = dp.ts;
      if (c.nt > 0) {                  // a lazy cut: locate its last kept tie first
        const uint32_t K = static_cast<uint32_t>(t2.cut >> 32);
        const int idx = find_nth_with_key<DT>(c.trow, K, static_cast<uint32_t>(c.nt), sm);
        t2.cut = composite(K, static_cast<uint32_t>(idx));
      }
      RowStat d0;
      d0.path = PATH_FULL; d0.W = 1.0; d0.cut = 0; d0.m = 0.0f; d0.n_list = 0; d0.cT = 0.0f; d0.invW = 1.0f;
      ScanCtx sc = make_scan<DT>(a, b, j, 0, onehot, t2, d0, -1, sm);
      double Zp;
      tok = block_scan_draw<DT>(sc, u, false, Zp, flags, sm);
    }
  } else {
    chunk_exact<DT, MODE>(c, a.chunk_vecs, dp.K, dp.Kbt, dp.Kbd, true, dp.tl, &tok, sm, wbuf);
  }
  if (tid == 0) {
    a.out_tokens[static_cast<size_t>(b) * (a.G + 1) + j] = tok;
    if (a.out_Z) a.out_Z[b] = mode != 0 ? static_cast<float>(Z) : -1.0f;
    if (a.eos >= 0 && tok == a.eos) flags |= SEQ_FLAG_EOS;
    if (a.out_status) a.out_status[b] = flags;
    a.dcount[b] = 0u;   // leave the workspace reusable
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 3) draw_kernel(const SampleArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  DrawPart& dp = *reinterpret_cast<DrawPart*>(smem_raw + sizeof(Smem));
  // launched as a programmatic dependent of the row kernel: its records are
  // read only once that grid has completed
  grid_dependency_wait();
  const int b = blockIdx.x;
  const DrawRec rec = a.drec[b];
  if (rec.j < 0) return;
  const int slots = 2 * a.G + 1;
  const bool onehot = a.dft == nullptr || (a.onehot != nullptr && a.onehot[b] != 0);
  const RowStat* S = a.stats + static_cast<size_t>(b) * slots;
  const RowStat ts = load_stat(S + rec.j);
  RowStat ds;
  ds.path = PATH_FULL; ds.W = 1.0; ds.cut = 0; ds.m = 0.0f; ds.n_list = 0; ds.cT = 0.0f; ds.invW = 1.0f;
  if (rec.mode != 0 && !onehot) ds = load_stat(S + a.G + 1 + rec.j);
  const uint32_t stage0 = smem_u32(smem_raw + kDrawStageOff);
  float* wbuf = reinterpret_cast<float*>(smem_raw + kDrawStageOff);
  switch (rec.mode) {
    case 0: draw_body<DT, 0>(a, b, rec, ts, ds, onehot, sm, dp, stage0, wbuf); break;
    case 1: draw_body<DT, 1>(a, b, rec, ts, ds, onehot, sm, dp, stage0, wbuf); break;
    case 2: draw_body<DT, 2>(a, b, rec, ts, ds, onehot, sm, dp, stage0, wbuf); break;
    default: draw_body<DT, 3>(a, b, rec, ts, ds, onehot, sm, dp, stage0, wbuf); break;
  }
}

// ------------------------------------------------------------------ greedy
struct GreedyArgs {
  const char* tgt;
  const int32_t* tokens;
  const int32_t* gammas;
  int B, G, V;
  int aligned;
  size_t row_bytes;
  uint32_t* counters;
  int2* rows;   // [B][G+1] (argmax, status)
  int32_t* out_tokens;
  int32_t* out_nacc;
  int32_t* out_status;
  int early_logits;   // the caller allows reading logits before the previous grid completes
};

template <int DT>
__global__ void __launch_bounds__(kThreads, 5) greedy_kernel(const GreedyArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  // a programmatic dependent of the previous call: with early logits reads
  // allowed and no per-sequence lengths every row is used, and a row CTA takes
  // its argmax before it waits for the previous grid (then reads tokens and
  // writes), so back-to-back calls overlap
  const bool stream_first = a.early_logits && a.gammas == nullptr;
  if (!stream_first) grid_dependency_wait();
  grid_launch_dependents();
  const int slots = a.G + 1;
  const int b = blockIdx.x / slots;
  const int i = blockIdx.x - b * slots;
  const int gb = a.gammas ? a.gammas[b] : a.G;
  const size_t ob = static_cast<size_t>(b) * (a.G + 1);
  if (gb < 0 || gb > a.G) {
    if (i == 0) {
      for (int t = threadIdx.x; t <= a.G; t += kThreads) a.out_tokens[ob + t] = -1;
      if (threadIdx.x == 0) {
        a.out_nacc[b] = -1;
        if (a.out_status) a.out_status[b] = SEQ_BAD_LENGTH;
      }
    }
    return;
  }
  if (i > gb) return;
  const Row row = make_row<DT>(a.tgt + (static_cast<size_t>(b) * slots + i) * a.row_bytes, a.V, a.aligned != 0);
  int g, st;
  greedy_row<DT>(row, sm, g, st);
  if (stream_first) grid_dependency_wait();
  if (threadIdx.x == 0) a.rows[static_cast<size_t>(b) * slots + i] = make_int2(g, st);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&a.counters[b], 1u);
    sm.b_i32[7] = (prev + 1u == static_cast<unsigned>(gb + 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!sm.b_i32[7]) return;
  __threadfence();
  if (threadIdx.x == 0) {
    // [wrblog §7.1]: accept while d_i == argmax p_i; emit argmax at the first mismatch
    int status = SEQ_OK;
    for (int k = 0; k < gb && status == SEQ_OK; ++k) {
      const int t = a.tokens[static_cast<size_t>(b) * a.G + k];
      if (t < 0 || t >= a.V) status = SEQ_BAD_TOKEN;
    }
    const int2* R = a.rows + static_cast<size_t>(b) * slots;
    for (int k = 0; k <= gb && status == SEQ_OK; ++k) status = __ldcg(&R[k].y);
    if (status != SEQ_OK) {
      for (int t = 0; t <= a.G; ++t) a.out_tokens[ob + t] = -1;
      a.out_nacc[b] = -1;
    } else {
      int j = gb;
      for (int k = 0; k < gb; ++k) {
        if (a.tokens[static_cast<size_t>(b) * a.G + k] != __ldcg(&R[k].x)) { j = k; break; }
      }
      for (int t = 0; t <= a.G; ++t) {
        int v = -1;
        if (t < j) v = a.tokens[static_cast<size_t>(b) * a.G + t];
        else if (t == j) v = __ldcg(&R[j].x);
        a.out_tokens[ob + t] = v;
      }
      a.out_nacc[b] = j;
    }
    if (a.out_status) a.out_status[b] = status;
    a.counters[b] = 0u;
  }
}

// ------------------------------------------------------------------ greedy tree
// Greedy verification of a draft tree [baisen §8; magicnet §7]: node 0 is the
// root, node i > 0 carries a draft token and a parent p_i < i, and target row
// i scores the token after the path root..i.  One CTA per node row computes
// its argmax; the last CTA of the sequence walks from the root, moving to the
// first child (in index order) whose token is the current node's argmax, and
// emits the argmax where no child matches.  Warp 0 does the checks and the
// walk: every step scans the candidate children 32 at a time with a ballot.
struct TreeArgs {
  const char* tgt;
  const int32_t* tokens;    // [B][N]
  const int32_t* parents;   // [B][N]
  const int32_t* nodes;     // [B] or null (N everywhere)
  int B, N, V;
  int aligned;
  size_t row_bytes;
  uint32_t* counters;       // [B]
  int2* rows;               // [B][N] (argmax, status)
  int32_t* out_tokens;      // [B][N]
  int32_t* out_nacc;        // [B]
  int32_t* out_path;        // [B][N] or null
  int32_t* out_status;      // [B] or null
  int early_logits;         // the caller allows reading logits before the previous grid completes
};

__device__ void tree_fail(const TreeArgs& a, int b, int status, int lane) {
  const size_t ob = static_cast<size_t>(b) * a.N;
  for (int t = lane; t < a.N; t += 32) {
    a.out_tokens[ob + t] = -1;
    if (a.out_path) a.out_path[ob + t] = -1;
  }
  if (lane == 0) {
    a.out_nacc[b] = -1;
    if (a.out_status) a.out_status[b] = status;
  }
}

template <int DT>
__global__ void __launch_bounds__(kThreads, 5) greedy_tree_kernel(const TreeArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  // as greedy_kernel: with early logits reads allowed and no per-sequence node
  // counts every node row is used and a CTA takes its argmax before waiting
  // for the previous grid
  const bool stream_first = a.early_logits && a.nodes == nullptr;
  if (!stream_first) grid_dependency_wait();
  grid_launch_dependents();
  const int b = blockIdx.x / a.N;
  const int i = blockIdx.x - b * a.N;
  const int n = a.nodes ? a.nodes[b] : a.N;
  const int lane = threadIdx.x & 31;
  if (n < 1 || n > a.N) {
    if (i == 0 && threadIdx.x < 32) tree_fail(a, b, SEQ_BAD_LENGTH, lane);
    return;
  }
  if (i >= n) return;
  const Row row = make_row<DT>(a.tgt + (static_cast<size_t>(b) * a.N + i) * a.row_bytes, a.V, a.aligned != 0);
  int g, st;
  greedy_row<DT>(row, sm, g, st);
  if (stream_first) grid_dependency_wait();
  if (threadIdx.x == 0) a.rows[static_cast<size_t>(b) * a.N + i] = make_int2(g, st);
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&a.counters[b], 1u);
    sm.b_i32[7] = (prev + 1u == static_cast<unsigned>(n)) ? 1 : 0;
  }
  __syncthreads();
  if (!sm.b_i32[7] || threadIdx.x >= 32) return;
  __threadfence();
  const size_t ob = static_cast<size_t>(b) * a.N;
  const int32_t* T = a.tokens + ob;
  const int32_t* Pa = a.parents + ob;
  const int2* R = a.rows + ob;
  // checks in the documented order: node tokens, parents, then the rows in node order
  int status = SEQ_OK;
  bool bad_tok = false, bad_par = false;
  for (int c = 1 + lane; c < n; c += 32) {
    bad_tok |= T[c] < 0 || T[c] >= a.V;
    bad_par |= Pa[c] < 0 || Pa[c] >= c;
  }
  if (__any_sync(kFull, bad_tok)) status = SEQ_BAD_TOKEN;
  else if (__any_sync(kFull, bad_par)) status = SEQ_BAD_TREE;
  for (int base = 0; base < n && status == SEQ_OK; base += 32) {
    const int st2 = base + lane < n ? __ldcg(&R[base + lane].y) : SEQ_OK;
    const unsigned m = __ballot_sync(kFull, st2 != SEQ_OK);
    if (m) status = __shfl_sync(kFull, st2, __ffs(m) - 1);
  }
  if (status != SEQ_OK) {
    tree_fail(a, b, status, lane);
    if (lane == 0) a.counters[b] = 0u;
    return;
  }
  // the walk: the first child of cur (index order) whose token is cur's argmax
  int cur = 0, L = 0;
  if (lane == 0 && a.out_path) a.out_path[ob] = 0;
  while (true) {
    const int gcur = __ldcg(&R[cur].x);
    int next = -1;
    for (int base = cur + 1; base < n && next < 0; base += 32) {
      const int c = base + lane;
      const unsigned m = __ballot_sync(kFull, c < n && Pa[c] == cur && T[c] == gcur);
      if (m) next = base + __ffs(m) - 1;
    }
    if (next < 0) {
      if (lane == 0) a.out_tokens[ob + L] = gcur;           // the correction, or the bonus at a leaf
      break;
    }
    if (lane == 0) {
      a.out_tokens[ob + L] = T[next];
      if (a.out_path) a.out_path[ob + L + 1] = next;
    }
    cur = next;
    ++L;
  }
  for (int t = L + 1 + lane; t < a.N; t += 32) {
    a.out_tokens[ob + t] = -1;
    if (a.out_path && t > L) a.out_path[ob + t] = -1;
  }
  if (lane == 0) {
    a.out_nacc[b] = L;
    if (a.out_status) a.out_status[b] = SEQ_OK;
    a.counters[b] = 0u;                                     // leave the workspace reusable
  }
}

// ------------------------------------------------------------------ early-exit greedy
// Greedy verification that stops at the first mismatch [wrblog §6, §7.1],
// without making any CTA wait for another.  The grid is position-major: CTA
// (i, b) analyses row i of sequence b, and all row-0 CTAs come first, then
// row 1, and so on, so a row's predecessors have usually finished by the time
// it is scheduled.  A CTA first reads its sequence's stop record; if an
// earlier row already failed or mismatched it skips its row without reading
// it.  Otherwise it analyses the row and, on a mismatch (or a failed row),
// lowers the stop record.  The last CTA of the sequence forms the result from
// rows 0..stop only, so a row read speculatively after the stop never affects
// it.  Stop records encode row s as G + 1 - s (0 = none) so that atomicMax
// keeps the earliest stop and a zero-filled workspace means "no stop".
//
// Rows whose predecessors are still running are read speculatively; each
// warp of such a row keeps watching the stop record and the row is abandoned
// (reported as not read) once an earlier row stops the sequence.  Making
// such a CTA wait (bounded) for the row a wave earlier cut the rows read from
// about 7.1 to 5.3 per sequence at greedy-at-scale sizes but made the launch
// slower (waiting CTAs hold slots, and the waves serialise), so nothing waits.
template <int DT>
__global__ void __launch_bounds__(kThreads, 5) greedy_early_kernel(const GreedyArgs a, uint32_t* stop_enc,
                                                                   int32_t* out_rows) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int i = blockIdx.x / a.B;
  const int b = blockIdx.x - i * a.B;
  const int slots = a.G + 1;
  const int gb = a.gammas ? a.gammas[b] : a.G;
  const size_t ob = static_cast<size_t>(b) * slots;
  const size_t tb = static_cast<size_t>(b) * a.G;
  if (gb < 0 || gb > a.G) {
    if (i == 0) {
      for (int t = threadIdx.x; t <= a.G; t += kThreads) a.out_tokens[ob + t] = -1;
      if (threadIdx.x == 0) {
        a.out_nacc[b] = -1;
        if (a.out_status) a.out_status[b] = SEQ_BAD_LENGTH;
        if (out_rows) out_rows[b] = 0;
      }
    }
    return;
  }
  if (i > gb) return;
  if (threadIdx.x == 0) {
    sm.b_i32[0] = static_cast<int>(__ldcg(&stop_enc[b]));
    sm.early_skip = 0;
  }
  __syncthreads();
  const bool skip = static_cast<uint32_t>(sm.b_i32[0]) > static_cast<uint32_t>(slots - i);   // a stop before row i
  int2 res = make_int2(-1, -1);   // (argmax, status); status -1 = row not read (or abandoned)
  if (!skip) {
    const Row row = make_row<DT>(a.tgt + (ob + i) * a.row_bytes, a.V, a.aligned != 0);
    StopCheck sc;                  // a stop before row i arriving meanwhile abandons the row
    if (i > 0) {
      sc.p = stop_enc + b;
      sc.thr = static_cast<unsigned>(slots - i);
    }
    int g, st;
    greedy_row<DT>(row, sm, g, st, sc);
    if (!sm.early_skip) {
      res = make_int2(g, st);
      if (threadIdx.x == 0 && (st != SEQ_OK || (i < gb && a.tokens[tb + i] != g)))
        atomicMax(&stop_enc[b], static_cast<uint32_t>(slots - i));
    }
  }
  if (threadIdx.x == 0) a.rows[ob + i] = res;
  __threadfence();
  __syncthreads();
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(&a.counters[b], 1u);
    sm.b_i32[7] = (prev + 1u == static_cast<unsigned>(gb + 1)) ? 1 : 0;
  }
  __syncthreads();
  if (!sm.b_i32[7]) return;
  __threadfence();
  if (threadIdx.x == 0) {
    // the documented order: tokens, then the rows up to the stop
    int status = SEQ_OK;
    for (int k = 0; k < gb && status == SEQ_OK; ++k) {
      const int t = a.tokens[tb + k];
      if (t < 0 || t >= a.V) status = SEQ_BAD_TOKEN;
    }
    const uint32_t se = __ldcg(&stop_enc[b]);
    const int j = se ? slots - static_cast<int>(se) : gb;   // rows 0..j-1 matched; row j was read
    const int2* R = a.rows + ob;
    int nread = 0;
    for (int k = 0; k <= gb; ++k) nread += __ldcg(&R[k].y) >= 0 ? 1 : 0;
    const int2 rj = __ldcg(&R[j]);
    if (status == SEQ_OK) status = rj.y;
    if (status != SEQ_OK) {
      for (int t = 0; t <= a.G; ++t) a.out_tokens[ob + t] = -1;
      a.out_nacc[b] = -1;
    } else {
      for (int t = 0; t <= a.G; ++t) {
        int v = -1;
        if (t < j) v = a.tokens[tb + t];
        else if (t == j) v = rj.x;
        a.out_tokens[ob + t] = v;
      }
      a.out_nacc[b] = j;
    }
    if (a.out_status) a.out_status[b] = status;
    if (out_rows) out_rows[b] = status == SEQ_BAD_TOKEN ? 0 : nread;
    a.counters[b] = 0u;   // leave the workspace reusable
    stop_enc[b] = 0u;
  }
}

// ------------------------------------------------------------------ transform (test hook)
template <int DT>
__global__ void __launch_bounds__(kThreads, 5) transform_kernel(const char* logits, int V, RowParams P,
                                                                 int aligned, size_t row_bytes,
                                                                 float* out, int32_t* out_status) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  Smem& sm = *reinterpret_cast<Smem*>(smem_raw);
  const int r = blockIdx.x;
  const Row row = make_row<DT>(logits + static_cast<size_t>(r) * row_bytes, V, aligned != 0);
  if (P.path == PATH_STREAM) stream_row<DT>(row, P, -1, sm);
  else full_row<DT>(row, P, -1, sm);
  const RowStat st = sm.st;
  float* o = out + static_cast<size_t>(r) * V;
  if (st.status != SEQ_OK || st.path == PATH_STREAM) {
    for (int x = threadIdx.x; x < V; x += kThreads) o[x] = 0.0f;
    __syncthreads();
    if (st.status == SEQ_OK)
      for (int e = threadIdx.x; e < st.n_list; e += kThreads) o[sm.list_tok[e]] = sm.list_ph[e];
  } else {
    const float invW = st.invW;
    const CutTest ct = cut_test(st.cut);
    for (int x = threadIdx.x; x < V; x += kThreads)
      o[x] = full_prob(load_elem<DT>(row.base, x), static_cast<uint32_t>(x), ct, st.m, P.cT, invW);
  }
  if (out_status && threadIdx.x == 0) out_status[r] = st.status;
}

}  // namespace sv

// ====================================================================== host
namespace {

using namespace sv;

constexpr size_t kAlign = 256;
inline size_t round_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

bool params_ok(const spec_sampling_params_t& p) { return rule_ok(p); }

RowParams make_row_params(const spec_sampling_params_t& p, int V, spec_dtype_t) { return row_params_of(p, V); }

bool aligned_to(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

size_t elem_bytes(spec_dtype_t dt) { return dt == SPEC_BF16 ? 2 : 4; }
int elems_per_vec(spec_dtype_t dt) { return dt == SPEC_BF16 ? 8 : 4; }


// Chunks per row of the full-row draw (float32 rows have the most vectors).
int draw_chunks(int V, spec_dtype_t dt) {
  const long long nvec = (static_cast<long long>(V) + elems_per_vec(dt) - 1) / elems_per_vec(dt);
  return static_cast<int>((nvec + kChunkVecs - 1) / kChunkVecs);
}

// Workspace: the two per-sequence counter arrays come first -- the only part
// that must be zero when a call starts (kernels leave them zero again).
struct SampleLayout {
  size_t counters, dcount, stop, pairx, stats, lists, drec, dsum, total;
};
// counters, draw counters, early-exit stop marks, early-exit exchange words
size_t zero_region_bytes(int B, int G) {
  return 3 * round_up(static_cast<size_t>(B) * sizeof(uint32_t)) +
         round_up(static_cast<size_t>(B) * G * sizeof(unsigned long long));
}
// tps / dps: that side's rules come per sequence, so its rows may take either path.
SampleLayout sample_layout(int B, int G, int V, const RowParams& tp, const RowParams& dp, bool tps = false,
                           bool dps = false) {
  SampleLayout L;
  const size_t slots = static_cast<size_t>(2 * G + 1);
  L.counters = 0;
  L.dcount = round_up(static_cast<size_t>(B) * sizeof(uint32_t));
  L.stop = 2 * L.dcount;
  L.pairx = 3 * L.dcount;
  L.stats = zero_region_bytes(B, G);
  L.lists = L.stats + round_up(static_cast<size_t>(B) * slots * sizeof(RowStat));
  const bool need_lists = tps || dps || tp.path == PATH_STREAM || dp.path == PATH_STREAM;
  L.drec = L.lists + (need_lists ? round_up(static_cast<size_t>(B) * slots * kListCap * sizeof(ListEntry)) : 0);
  const bool defer = tps || tp.path == PATH_FULL;
  L.dsum = L.drec + (defer ? round_up(static_cast<size_t>(B) * sizeof(DrawRec)) : 0);
  L.total = L.dsum + (defer ? round_up(static_cast<size_t>(B) * draw_chunks(V, SPEC_F32) * sizeof(ChunkSum)) : 0);
  return L;
}

// Greedy workspace: per-sequence counters and stop records first (the part that
// must start at zero; kernels leave it zero), then the per-row (argmax, status).
struct GreedyLayout {
  size_t counters, stop, rows, total;
};
GreedyLayout greedy_layout(int B, int G) {
  GreedyLayout L;
  const size_t cb = round_up(static_cast<size_t>(B) * sizeof(uint32_t));
  L.counters = 0;
  L.stop = cb;
  L.rows = 2 * cb;
  L.total = L.rows + round_up(static_cast<size_t>(B) * (G + 1) * sizeof(int2));
  return L;
}

bool shape_ok(int B, int G, int V) {
  if (B < 1 || G < 0 || V < 1) return false;
  const long long slots = 2LL * G + 1;
  return static_cast<long long>(B) * slots <= 0x7fffffffLL;
}

// Raises a kernel's dynamic shared memory limit once per device (the attribute
// is per device; later calls only read an atomic bit mask).
template <typename K>
cudaError_t prepare(K kernel, std::atomic<uint64_t>& done, size_t smem = sizeof(Smem) + sizeof(FullExtra)) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  const uint64_t bit = 1ull << (dev & 63);
  if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
  err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
  if (err == cudaSuccess) done.fetch_or(bit, std::memory_order_acq_rel);
  return err;
}
// The kernels' status codes are the header's.
static_assert(int(SEQ_OK) == int(SPEC_SEQ_OK) && int(SEQ_BAD_LENGTH) == int(SPEC_SEQ_BAD_LENGTH) &&
              int(SEQ_BAD_TOKEN) == int(SPEC_SEQ_BAD_TOKEN) && int(SEQ_BAD_UNIFORM) == int(SPEC_SEQ_BAD_UNIFORM) &&
              int(SEQ_NONFINITE) == int(SPEC_SEQ_NONFINITE) && int(SEQ_EMPTY_SUPPORT) == int(SPEC_SEQ_EMPTY_SUPPORT) &&
              int(SEQ_BAD_PARAMS) == int(SPEC_SEQ_BAD_PARAMS) && int(SEQ_BAD_TREE) == int(SPEC_SEQ_BAD_TREE) &&
              int(SEQ_STALLED) == int(SPEC_SEQ_STALLED) && int(SEQ_FLAG_ZERO_Q) == int(SPEC_SEQ_FLAG_ZERO_Q) &&
              int(SEQ_FLAG_Z_ZERO) == int(SPEC_SEQ_FLAG_Z_ZERO) && int(SEQ_FLAG_EOS) == int(SPEC_SEQ_FLAG_EOS),
              "status codes");

std::atomic<uint64_t> g_ready[18];
std::atomic<int> g_early_logits{0};   // spec_set_early_logits_reads  // sample, greedy, transform, draw, greedy-early, sample-ex, tree, kept-list, sample-tree x {bf16, f32}

// Streaming multiprocessors of the current device (cached per device).
int sm_count() {
  static std::atomic<int> cache[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 1;
  const int d = dev & 63;
  int n = cache[d].load(std::memory_order_relaxed);
  if (n > 0) return n;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n < 1) n = 1;
  cache[d].store(n, std::memory_order_relaxed);
  return n;
}

// Chunks per draw CTA: about two waves of three draw CTAs per SM over the
// batch, each CTA summing at least one and at most kDrawMaxRun chunks.
int draw_run(int B, int nchunk) {
  const int target = 2 * 3 * sm_count();
  int splits = std::max(1, std::min(nchunk, (target + B - 1) / B));
  splits = std::max(splits, (nchunk + kDrawMaxRun - 1) / kDrawMaxRun);
  return (nchunk + splits - 1) / splits;
}

// A launch as a programmatic dependent of the previous kernel in the stream
// (the kernel waits for that grid itself before it reads anything the grid
// may have written).
template <typename K, typename Arg>
cudaError_t launch_pdl(K kernel, dim3 grid, size_t smem, cudaStream_t s, const Arg& arg) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, arg);
}

// The full-row draw, as a programmatic dependent of the row kernel (it waits
// for that grid before reading its records; launching early hides the gap).
template <typename K>
cudaError_t launch_draw(K kernel, const SampleArgs& a, dim3 grid, cudaStream_t s) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kDrawSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, a);
}


// Dynamic shared memory of a launch: the bracketing top-p of PATH_FULL rows
// needs FullExtra after Smem; launches without such rows keep their occupancy.
size_t smem_for(const RowParams& a, const RowParams& b, spec_dtype_t dt) {
  auto topp_full = [](const RowParams& r) { return r.path == PATH_FULL && r.top_p < 1.0f; };
  if (!topp_full(a) && !topp_full(b)) return sizeof(Smem);
  // bf16 top-p rows without top-k take the value counts, which use only the
  // count tables (four CTAs per SM); any other full-row top-p row brackets
  auto counts_only = [&](const RowParams& r) { return !topp_full(r) || (dt == SPEC_BF16 && r.k == 0); };
  return sizeof(Smem) + ((counts_only(a) && counts_only(b)) ? kKCExtraBytes : sizeof(FullExtra));
}

}  // namespace

extern "C" {

spec_status_t spec_set_early_logits_reads(int32_t enable) {
  g_early_logits.store(enable != 0 ? 1 : 0, std::memory_order_relaxed);
  return SPEC_OK;
}

const char* spec_status_string(spec_status_t s) {
  switch (s) {
    case SPEC_OK: return "ok";
    case SPEC_ERR_INVALID_ARG: return "invalid argument";
    case SPEC_ERR_UNSUPPORTED: return "unsupported request";
    case SPEC_ERR_MISALIGNED: return "misaligned pointer";
    case SPEC_ERR_WORKSPACE: return "workspace too small";
    case SPEC_ERR_CUDA: return "CUDA runtime error";
  }
  return "unknown status";
}

spec_status_t spec_verify_workspace_size(int32_t batch, int32_t gamma_max, int32_t vocab,
                                         spec_sampling_params_t target_params,
                                         spec_sampling_params_t draft_params, size_t* bytes) {
  if (!bytes || !shape_ok(batch, gamma_max, vocab) || !params_ok(target_params) || !params_ok(draft_params))
    return SPEC_ERR_INVALID_ARG;
  if (gamma_max > kMaxGamma) return SPEC_ERR_UNSUPPORTED;
  *bytes = sample_layout(batch, gamma_max, vocab, make_row_params(target_params, vocab, SPEC_BF16),
                         make_row_params(draft_params, vocab, SPEC_BF16)).total;
  return SPEC_OK;
}

spec_status_t spec_verify_workspace_size_ex(int32_t batch, int32_t gamma_max, int32_t vocab,
                                            spec_sampling_params_t target_params,
                                            spec_sampling_params_t draft_params,
                                            const spec_verify_options_t* options, size_t* bytes) {
  if (!bytes || !shape_ok(batch, gamma_max, vocab) || !params_ok(target_params) || !params_ok(draft_params))
    return SPEC_ERR_INVALID_ARG;
  if (gamma_max > kMaxGamma) return SPEC_ERR_UNSUPPORTED;
  const bool tps = options && options->target_params_seq, dps = options && options->draft_params_seq;
  const bool any_path = !(options && options->kept_list_only);
  *bytes = sample_layout(batch, gamma_max, vocab, make_row_params(target_params, vocab, SPEC_BF16),
                         make_row_params(draft_params, vocab, SPEC_BF16), any_path && tps, any_path && dps).total;
  return SPEC_OK;
}

spec_status_t spec_greedy_workspace_size(int32_t batch, int32_t gamma_max, size_t* bytes) {
  if (!bytes || !shape_ok(batch, gamma_max, 1)) return SPEC_ERR_INVALID_ARG;
  *bytes = greedy_layout(batch, gamma_max).total;
  return SPEC_OK;
}

// spec_verify_sample and spec_verify_sample_lenient: one body, beta = lenience.
static spec_status_t verify_sample_impl(const void* target_logits, const void* draft_logits,
                                        spec_dtype_t dtype, const int32_t* draft_tokens,
                                        const int32_t* gamma_per_seq, const uint8_t* draft_is_onehot,
                                        const float* u_accept, const float* u_sample,
                                        spec_sampling_params_t target_params,
                                        spec_sampling_params_t draft_params,
                                        const spec_verify_options_t* options,
                                        int32_t batch, int32_t gamma_max, int32_t vocab,
                                        void* workspace, size_t workspace_bytes,
                                        int32_t* out_tokens, int32_t* out_num_accepted,
                                        float* out_accept_prob, float* out_residual_z,
                                        int32_t* out_status, int32_t* out_num_emitted, void* stream,
                                        bool clear_zero_region = false) {
  if (dtype != SPEC_BF16 && dtype != SPEC_F32) return SPEC_ERR_INVALID_ARG;
  const float lenience = options ? options->lenience : 1.0f;
  const int32_t eos = options ? options->eos_token : -1;
  const spec_sampling_params_t* tps = options ? options->target_params_seq : nullptr;
  const spec_sampling_params_t* dps = options ? options->draft_params_seq : nullptr;
  const bool kept_only = options && options->kept_list_only && (tps || dps);
  const bool early = options && options->early_exit;
  if (!(lenience > 0.0f && lenience <= 1.0f)) return SPEC_ERR_INVALID_ARG;
  if (eos < -1 || eos >= vocab) return SPEC_ERR_INVALID_ARG;
  if (!aligned_to(tps, 4) || !aligned_to(dps, 4) || !aligned_to(out_num_emitted, 4)) return SPEC_ERR_MISALIGNED;
  if (!shape_ok(batch, gamma_max, vocab) || !params_ok(target_params) || !params_ok(draft_params))
    return SPEC_ERR_INVALID_ARG;
  if (gamma_max > kMaxGamma) return SPEC_ERR_UNSUPPORTED;
  if (!target_logits || !u_sample || !out_tokens || !out_num_accepted || !workspace) return SPEC_ERR_INVALID_ARG;
  if (gamma_max > 0 && (!draft_tokens || !u_accept)) return SPEC_ERR_INVALID_ARG;
  const size_t es = elem_bytes(dtype);
  if (!aligned_to(target_logits, es) || (draft_logits && !aligned_to(draft_logits, es)) ||
      !aligned_to(draft_tokens, 4) || !aligned_to(gamma_per_seq, 4) || !aligned_to(u_accept, 4) ||
      !aligned_to(u_sample, 4) || !aligned_to(out_tokens, 4) || !aligned_to(out_num_accepted, 4) ||
      !aligned_to(out_accept_prob, 4) || !aligned_to(out_residual_z, 4) || !aligned_to(out_status, 4) ||
      !aligned_to(workspace, kAlign))
    return SPEC_ERR_MISALIGNED;
  SampleArgs a;
  a.early_logits = g_early_logits.load(std::memory_order_relaxed);
  a.fast = nullptr;
  a.wpr = 0;
  a.tp = make_row_params(target_params, vocab, dtype);
  a.dp = make_row_params(draft_params, vocab, dtype);
  // promised kept-list rules: the scalar rules must keep the promise too
  if (kept_only && (a.tp.path != PATH_STREAM || a.dp.path != PATH_STREAM)) return SPEC_ERR_INVALID_ARG;
  const bool any_path = !kept_only && (tps || dps);     // per-sequence rows may take either path
  const SampleLayout L = sample_layout(batch, gamma_max, vocab, a.tp, a.dp, any_path && tps, any_path && dps);
  if (workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  a.tps = tps;
  a.dps = dps;
  a.eos = eos;
  a.kept_only = kept_only ? 1 : 0;
  a.out_nemit = out_num_emitted;
  a.tgt = static_cast<const char*>(target_logits);
  a.dft = static_cast<const char*>(draft_logits);
  a.tokens = draft_tokens;
  a.gammas = gamma_per_seq;
  a.onehot = draft_is_onehot;
  a.u_acc = u_accept;
  a.u_samp = u_sample;
  a.beta = lenience;
  a.B = batch;
  a.G = gamma_max;
  a.V = vocab;
  a.aligned = (vocab % elems_per_vec(dtype) == 0) && aligned_to(target_logits, 16) &&
              (!draft_logits || aligned_to(draft_logits, 16));
  a.row_bytes = static_cast<size_t>(vocab) * es;
  a.counters = reinterpret_cast<uint32_t*>(ws + L.counters);
  a.stats = reinterpret_cast<RowStat*>(ws + L.stats);
  a.lists = reinterpret_cast<ListEntry*>(ws + L.lists);
  a.out_tokens = out_tokens;
  a.out_nacc = out_num_accepted;
  a.out_aprob = out_accept_prob;
  a.out_Z = out_residual_z;
  a.out_status = out_status;
  a.defer = ((any_path && tps) || a.tp.path == PATH_FULL) ? 1 : 0;
  // per-sequence rules: any row may take the full-row path with a top-p cut
  const size_t smem = any_path ? sizeof(Smem) + sizeof(FullExtra) : smem_for(a.tp, a.dp, dtype);
  a.chunk_vecs = kChunkVecs;
  a.nchunk = draw_chunks(vocab, dtype);
  a.dcount = reinterpret_cast<uint32_t*>(ws + L.dcount);
  a.drec = reinterpret_cast<DrawRec*>(ws + L.drec);
  a.dsum = reinterpret_cast<ChunkSum*>(ws + L.dsum);
  a.early = early ? 1 : 0;
  a.stop_enc = reinterpret_cast<uint32_t*>(ws + L.stop);
  a.pairx = reinterpret_cast<unsigned long long*>(ws + L.pairx);
  // early exit: position-major, two CTA slots (target, draft) per sequence and position
  const unsigned grid = early ? static_cast<unsigned>(batch) * 2u * static_cast<unsigned>(gamma_max + 1)
                              : static_cast<unsigned>(batch) * static_cast<unsigned>(2 * gamma_max + 1);
  a.draw_run = draw_run(batch, a.nchunk);
  const dim3 dgrid(static_cast<unsigned>(batch), static_cast<unsigned>((a.nchunk + a.draw_run - 1) / a.draw_run));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err;
  // every host check has passed: a caller-less scratch gets its counters cleared
  // on the stream, right before the launches
  if (clear_zero_region && cudaMemsetAsync(workspace, 0, zero_region_bytes(batch, gamma_max), s) != cudaSuccess)
    return SPEC_ERR_CUDA;
  const bool ex = tps || dps || eos >= 0 || out_num_emitted || early;
  // the kept-list kernel: every used row on the streaming top-k path, aligned
  // rows, and each sequence's row blocks within the epilogue's gather buffer
  const int kcap = std::max(a.tp.k, draft_logits ? a.dp.k : 0);
  const bool list_path = !ex && a.aligned && a.tp.path == PATH_STREAM &&
                         (draft_logits == nullptr || a.dp.path == PATH_STREAM) && gamma_max <= 31 &&
                         (2 * gamma_max + 1) * (1 + kcap) <= kGatherWords;
  if (list_path) {
    a.fast = reinterpret_cast<uint4*>(ws + L.stats);
    a.wpr = 1 + kcap;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = sizeof(Smem);
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (dtype == SPEC_BF16) {
      err = prepare(sample_list_kernel<DT_BF16>, g_ready[14]);
      if (err == cudaSuccess) err = cudaLaunchKernelEx(&cfg, sample_list_kernel<DT_BF16>, a);
    } else {
      err = prepare(sample_list_kernel<DT_F32>, g_ready[15]);
      if (err == cudaSuccess) err = cudaLaunchKernelEx(&cfg, sample_list_kernel<DT_F32>, a);
    }
  } else if (dtype == SPEC_BF16 && ex) {
    err = prepare(sample_kernel<DT_BF16, true>, g_ready[10]);
    if (err == cudaSuccess) sample_kernel<DT_BF16, true><<<grid, kThreads, smem, s>>>(a);
    if (err == cudaSuccess && a.defer) err = prepare(draw_kernel<DT_BF16>, g_ready[6], kDrawSmem);
    if (err == cudaSuccess && a.defer) err = launch_draw(draw_kernel<DT_BF16>, a, dgrid, s);
  } else if (ex) {
    err = prepare(sample_kernel<DT_F32, true>, g_ready[11]);
    if (err == cudaSuccess) sample_kernel<DT_F32, true><<<grid, kThreads, smem, s>>>(a);
    if (err == cudaSuccess && a.defer) err = prepare(draw_kernel<DT_F32>, g_ready[7], kDrawSmem);
    if (err == cudaSuccess && a.defer) err = launch_draw(draw_kernel<DT_F32>, a, dgrid, s);
  } else if (dtype == SPEC_BF16) {
    err = prepare(sample_kernel<DT_BF16, false>, g_ready[0]);
    if (err == cudaSuccess) sample_kernel<DT_BF16, false><<<grid, kThreads, smem, s>>>(a);
    if (err == cudaSuccess && a.defer) err = prepare(draw_kernel<DT_BF16>, g_ready[6], kDrawSmem);
    if (err == cudaSuccess && a.defer) err = launch_draw(draw_kernel<DT_BF16>, a, dgrid, s);
  } else {
    err = prepare(sample_kernel<DT_F32, false>, g_ready[1]);
    if (err == cudaSuccess) sample_kernel<DT_F32, false><<<grid, kThreads, smem, s>>>(a);
    if (err == cudaSuccess && a.defer) err = prepare(draw_kernel<DT_F32>, g_ready[7], kDrawSmem);
    if (err == cudaSuccess && a.defer) err = launch_draw(draw_kernel<DT_F32>, a, dgrid, s);
  }
  if (err == cudaSuccess) err = cudaGetLastError();
  return err == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t spec_verify_sample(const void* target_logits, const void* draft_logits,
                                 spec_dtype_t dtype, const int32_t* draft_tokens,
                                 const int32_t* gamma_per_seq, const uint8_t* draft_is_onehot,
                                 const float* u_accept, const float* u_sample,
                                 spec_sampling_params_t target_params,
                                 spec_sampling_params_t draft_params,
                                 int32_t batch, int32_t gamma_max, int32_t vocab,
                                 void* workspace, size_t workspace_bytes,
                                 int32_t* out_tokens, int32_t* out_num_accepted,
                                 float* out_accept_prob, float* out_residual_z,
                                 int32_t* out_status, void* stream) {
  return verify_sample_impl(target_logits, draft_logits, dtype, draft_tokens, gamma_per_seq,
                            draft_is_onehot, u_accept, u_sample, target_params, draft_params, nullptr,
                            batch, gamma_max, vocab, workspace, workspace_bytes, out_tokens,
                            out_num_accepted, out_accept_prob, out_residual_z, out_status, nullptr, stream);
}

spec_status_t spec_verify_sample_lenient(const void* target_logits, const void* draft_logits,
                                         spec_dtype_t dtype, const int32_t* draft_tokens,
                                         const int32_t* gamma_per_seq, const uint8_t* draft_is_onehot,
                                         const float* u_accept, const float* u_sample,
                                         spec_sampling_params_t target_params,
                                         spec_sampling_params_t draft_params, float lenience,
                                         int32_t batch, int32_t gamma_max, int32_t vocab,
                                         void* workspace, size_t workspace_bytes,
                                         int32_t* out_tokens, int32_t* out_num_accepted,
                                         float* out_accept_prob, float* out_residual_z,
                                         int32_t* out_status, void* stream) {
  spec_verify_options_t opt;
  opt.lenience = lenience;
  opt.eos_token = -1;
  opt.target_params_seq = nullptr;
  opt.draft_params_seq = nullptr;
  opt.kept_list_only = 0;
  opt.early_exit = 0;
  return verify_sample_impl(target_logits, draft_logits, dtype, draft_tokens, gamma_per_seq,
                            draft_is_onehot, u_accept, u_sample, target_params, draft_params, &opt,
                            batch, gamma_max, vocab, workspace, workspace_bytes, out_tokens,
                            out_num_accepted, out_accept_prob, out_residual_z, out_status, nullptr, stream);
}

spec_status_t spec_verify_sample_ex(const void* target_logits, const void* draft_logits,
                                    spec_dtype_t dtype, const int32_t* draft_tokens,
                                    const int32_t* gamma_per_seq, const uint8_t* draft_is_onehot,
                                    const float* u_accept, const float* u_sample,
                                    spec_sampling_params_t target_params,
                                    spec_sampling_params_t draft_params,
                                    const spec_verify_options_t* options,
                                    int32_t batch, int32_t gamma_max, int32_t vocab,
                                    void* workspace, size_t workspace_bytes,
                                    int32_t* out_tokens, int32_t* out_num_accepted,
                                    float* out_accept_prob, float* out_residual_z,
                                    int32_t* out_status, int32_t* out_num_emitted, void* stream) {
  return verify_sample_impl(target_logits, draft_logits, dtype, draft_tokens, gamma_per_seq,
                            draft_is_onehot, u_accept, u_sample, target_params, draft_params, options,
                            batch, gamma_max, vocab, workspace, workspace_bytes, out_tokens,
                            out_num_accepted, out_accept_prob, out_residual_z, out_status, out_num_emitted,
                            stream);
}

spec_status_t spec_tree_workspace_size(int32_t batch, int32_t max_nodes, size_t* bytes) {
  if (!bytes || max_nodes < 1 || !shape_ok(batch, max_nodes - 1, 1)) return SPEC_ERR_INVALID_ARG;
  *bytes = greedy_layout(batch, max_nodes - 1).total;     // counters, then [B][N] (argmax, status)
  return SPEC_OK;
}

spec_status_t spec_verify_greedy_tree(const void* target_logits, spec_dtype_t dtype,
                                      const int32_t* tree_tokens, const int32_t* tree_parents,
                                      const int32_t* nodes_per_seq, int32_t batch, int32_t max_nodes,
                                      int32_t vocab, void* workspace, size_t workspace_bytes,
                                      int32_t* out_tokens, int32_t* out_num_accepted, int32_t* out_path,
                                      int32_t* out_status, void* stream) {
  if (dtype != SPEC_BF16 && dtype != SPEC_F32) return SPEC_ERR_INVALID_ARG;
  if (max_nodes < 1 || vocab < 1 || !shape_ok(batch, max_nodes - 1, vocab)) return SPEC_ERR_INVALID_ARG;
  if (!target_logits || !tree_tokens || !tree_parents || !out_tokens || !out_num_accepted || !workspace)
    return SPEC_ERR_INVALID_ARG;
  const size_t es = elem_bytes(dtype);
  if (!aligned_to(target_logits, es) || !aligned_to(tree_tokens, 4) || !aligned_to(tree_parents, 4) ||
      !aligned_to(nodes_per_seq, 4) || !aligned_to(out_tokens, 4) || !aligned_to(out_num_accepted, 4) ||
      !aligned_to(out_path, 4) || !aligned_to(out_status, 4) || !aligned_to(workspace, kAlign))
    return SPEC_ERR_MISALIGNED;
  size_t need = 0;
  spec_tree_workspace_size(batch, max_nodes, &need);
  if (workspace_bytes < need) return SPEC_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  const GreedyLayout L = greedy_layout(batch, max_nodes - 1);
  TreeArgs a;
  a.early_logits = g_early_logits.load(std::memory_order_relaxed);
  a.tgt = static_cast<const char*>(target_logits);
  a.tokens = tree_tokens;
  a.parents = tree_parents;
  a.nodes = nodes_per_seq;
  a.B = batch;
  a.N = max_nodes;
  a.V = vocab;
  a.aligned = (vocab % elems_per_vec(dtype) == 0) && aligned_to(target_logits, 16);
  a.row_bytes = static_cast<size_t>(vocab) * es;
  a.counters = reinterpret_cast<uint32_t*>(ws + L.counters);
  a.rows = reinterpret_cast<int2*>(ws + L.rows);
  a.out_tokens = out_tokens;
  a.out_nacc = out_num_accepted;
  a.out_path = out_path;
  a.out_status = out_status;
  const unsigned grid = static_cast<unsigned>(batch) * static_cast<unsigned>(max_nodes);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (dtype == SPEC_BF16) {
    err = prepare(greedy_tree_kernel<DT_BF16>, g_ready[12]);
    if (err == cudaSuccess) err = launch_pdl(greedy_tree_kernel<DT_BF16>, dim3(grid), sizeof(Smem), s, a);
  } else {
    err = prepare(greedy_tree_kernel<DT_F32>, g_ready[13]);
    if (err == cudaSuccess) err = launch_pdl(greedy_tree_kernel<DT_F32>, dim3(grid), sizeof(Smem), s, a);
  }
  if (err == cudaSuccess) err = cudaGetLastError();
  return err == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

// Sampling tree workspace: per-sequence counters, then [B][2N] row blocks of
// wpr 16-byte words (a ListRec and the kept list).
constexpr int kMaxTreeNodes = 32;
struct TreeSampleLayout {
  size_t counters, blocks, total;
  int wpr;
};
bool tree_sample_layout(int B, int N, int V, const spec_sampling_params_t& tp, const spec_sampling_params_t& dp,
                        TreeSampleLayout& L, spec_status_t& why) {
  why = SPEC_ERR_INVALID_ARG;
  if (B < 1 || N < 1 || V < 1 || !params_ok(tp) || !params_ok(dp)) return false;
  if (static_cast<long long>(B) * 2 * N > 0x7fffffffLL) return false;
  why = SPEC_ERR_UNSUPPORTED;
  if (N > kMaxTreeNodes) return false;
  const RowParams t = row_params_of(tp, V), d = row_params_of(dp, V);
  if (t.path != PATH_STREAM || d.path != PATH_STREAM) return false;   // kept-list rules only
  L.wpr = 1 + std::max(t.k, d.k);
  L.counters = 0;
  L.blocks = round_up(static_cast<size_t>(B) * sizeof(uint32_t));
  L.total = L.blocks + round_up(static_cast<size_t>(B) * 2 * N * L.wpr * sizeof(uint4));
  return true;
}

spec_status_t spec_tree_sample_workspace_size(int32_t batch, int32_t max_nodes, int32_t vocab,
                                              spec_sampling_params_t target_params,
                                              spec_sampling_params_t draft_params, size_t* bytes) {
  if (!bytes) return SPEC_ERR_INVALID_ARG;
  TreeSampleLayout L;
  spec_status_t why;
  if (!tree_sample_layout(batch, max_nodes, vocab, target_params, draft_params, L, why)) return why;
  *bytes = L.total;
  return SPEC_OK;
}

spec_status_t spec_verify_sample_tree(const void* target_logits, const void* draft_logits, spec_dtype_t dtype,
                                      const int32_t* tree_tokens, const int32_t* tree_parents,
                                      const int32_t* nodes_per_seq, const float* u_node, const float* u_sample,
                                      spec_sampling_params_t target_params, spec_sampling_params_t draft_params,
                                      int32_t batch, int32_t max_nodes, int32_t vocab, void* workspace,
                                      size_t workspace_bytes, int32_t* out_tokens, int32_t* out_num_accepted,
                                      int32_t* out_path, float* out_accept_prob, float* out_residual_z,
                                      int32_t* out_status, void* stream) {
  if (dtype != SPEC_BF16 && dtype != SPEC_F32) return SPEC_ERR_INVALID_ARG;
  TreeSampleLayout L;
  spec_status_t why;
  if (!tree_sample_layout(batch, max_nodes, vocab, target_params, draft_params, L, why)) return why;
  if (!target_logits || !draft_logits || !tree_tokens || !tree_parents || !u_node || !u_sample || !out_tokens ||
      !out_num_accepted || !workspace)
    return SPEC_ERR_INVALID_ARG;
  const size_t es = elem_bytes(dtype);
  if (!aligned_to(target_logits, es) || !aligned_to(draft_logits, es) || !aligned_to(tree_tokens, 4) ||
      !aligned_to(tree_parents, 4) || !aligned_to(nodes_per_seq, 4) || !aligned_to(u_node, 4) ||
      !aligned_to(u_sample, 4) || !aligned_to(out_tokens, 4) || !aligned_to(out_num_accepted, 4) ||
      !aligned_to(out_path, 4) || !aligned_to(out_accept_prob, 4) || !aligned_to(out_residual_z, 4) ||
      !aligned_to(out_status, 4) || !aligned_to(workspace, kAlign))
    return SPEC_ERR_MISALIGNED;
  if (workspace_bytes < L.total) return SPEC_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  SampleTreeArgs a;
  a.early_logits = g_early_logits.load(std::memory_order_relaxed);
  a.tgt = static_cast<const char*>(target_logits);
  a.dft = static_cast<const char*>(draft_logits);
  a.tokens = tree_tokens;
  a.parents = tree_parents;
  a.nodes = nodes_per_seq;
  a.u_node = u_node;
  a.u_samp = u_sample;
  a.tp = make_row_params(target_params, vocab, dtype);
  a.dp = make_row_params(draft_params, vocab, dtype);
  a.B = batch;
  a.N = max_nodes;
  a.V = vocab;
  a.aligned = (vocab % elems_per_vec(dtype) == 0) && aligned_to(target_logits, 16) && aligned_to(draft_logits, 16);
  a.row_bytes = static_cast<size_t>(vocab) * es;
  a.counters = reinterpret_cast<uint32_t*>(ws + L.counters);
  a.blocks = reinterpret_cast<uint4*>(ws + L.blocks);
  a.wpr = L.wpr;
  a.out_tokens = out_tokens;
  a.out_nacc = out_num_accepted;
  a.out_path = out_path;
  a.out_aprob = out_accept_prob;
  a.out_Z = out_residual_z;
  a.out_status = out_status;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(batch) * 2u * static_cast<unsigned>(max_nodes));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = sizeof(Smem);
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  cudaError_t err;
  if (dtype == SPEC_BF16) {
    err = prepare(sample_tree_kernel<DT_BF16>, g_ready[16]);
    if (err == cudaSuccess) err = cudaLaunchKernelEx(&cfg, sample_tree_kernel<DT_BF16>, a);
  } else {
    err = prepare(sample_tree_kernel<DT_F32>, g_ready[17]);
    if (err == cudaSuccess) err = cudaLaunchKernelEx(&cfg, sample_tree_kernel<DT_F32>, a);
  }
  if (err == cudaSuccess) err = cudaGetLastError();
  return err == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t spec_verify_greedy(const void* target_logits, spec_dtype_t dtype,
                                 const int32_t* draft_tokens, const int32_t* gamma_per_seq,
                                 int32_t batch, int32_t gamma_max, int32_t vocab,
                                 void* workspace, size_t workspace_bytes,
                                 int32_t* out_tokens, int32_t* out_num_accepted,
                                 int32_t* out_status, void* stream) {
  if (dtype != SPEC_BF16 && dtype != SPEC_F32) return SPEC_ERR_INVALID_ARG;
  if (!shape_ok(batch, gamma_max, vocab)) return SPEC_ERR_INVALID_ARG;
  if (!target_logits || !out_tokens || !out_num_accepted || !workspace) return SPEC_ERR_INVALID_ARG;
  if (gamma_max > 0 && !draft_tokens) return SPEC_ERR_INVALID_ARG;
  const size_t es = elem_bytes(dtype);
  if (!aligned_to(target_logits, es) || !aligned_to(draft_tokens, 4) || !aligned_to(gamma_per_seq, 4) ||
      !aligned_to(out_tokens, 4) || !aligned_to(out_num_accepted, 4) || !aligned_to(out_status, 4) ||
      !aligned_to(workspace, kAlign))
    return SPEC_ERR_MISALIGNED;
  size_t need = 0;
  spec_greedy_workspace_size(batch, gamma_max, &need);
  if (workspace_bytes < need) return SPEC_ERR_WORKSPACE;
  char* ws = static_cast<char*>(workspace);
  GreedyArgs a;
  a.early_logits = g_early_logits.load(std::memory_order_relaxed);
  a.tgt = static_cast<const char*>(target_logits);
  a.tokens = draft_tokens;
  a.gammas = gamma_per_seq;
  a.B = batch;
  a.G = gamma_max;
  a.V = vocab;
  a.aligned = (vocab % elems_per_vec(dtype) == 0) && aligned_to(target_logits, 16);
  a.row_bytes = static_cast<size_t>(vocab) * es;
  const GreedyLayout L = greedy_layout(batch, gamma_max);
  a.counters = reinterpret_cast<uint32_t*>(ws + L.counters);
  a.rows = reinterpret_cast<int2*>(ws + L.rows);
  a.out_tokens = out_tokens;
  a.out_nacc = out_num_accepted;
  a.out_status = out_status;
  const unsigned grid = static_cast<unsigned>(batch) * static_cast<unsigned>(gamma_max + 1);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (dtype == SPEC_BF16) {
    err = prepare(greedy_kernel<DT_BF16>, g_ready[2]);
    if (err == cudaSuccess) err = launch_pdl(greedy_kernel<DT_BF16>, dim3(grid), sizeof(Smem), s, a);
  } else {
    err = prepare(greedy_kernel<DT_F32>, g_ready[3]);
    if (err == cudaSuccess) err = launch_pdl(greedy_kernel<DT_F32>, dim3(grid), sizeof(Smem), s, a);
  }
  if (err == cudaSuccess) err = cudaGetLastError();
  return err == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t spec_verify_greedy_early(const void* target_logits, spec_dtype_t dtype,
                                       const int32_t* draft_tokens, const int32_t* gamma_per_seq,
                                       int32_t batch, int32_t gamma_max, int32_t vocab,
                                       void* workspace, size_t workspace_bytes,
                                       int32_t* out_tokens, int32_t* out_num_accepted,
                                       int32_t* out_status, int32_t* out_rows_read, void* stream) {
  if (dtype != SPEC_BF16 && dtype != SPEC_F32) return SPEC_ERR_INVALID_ARG;
  if (!shape_ok(batch, gamma_max, vocab)) return SPEC_ERR_INVALID_ARG;
  if (!target_logits || !out_tokens || !out_num_accepted || !workspace) return SPEC_ERR_INVALID_ARG;
  if (gamma_max > 0 && !draft_tokens) return SPEC_ERR_INVALID_ARG;
  const size_t es = elem_bytes(dtype);
  if (!aligned_to(target_logits, es) || !aligned_to(draft_tokens, 4) || !aligned_to(gamma_per_seq, 4) ||
      !aligned_to(out_tokens, 4) || !aligned_to(out_num_accepted, 4) || !aligned_to(out_status, 4) ||
      !aligned_to(out_rows_read, 4) || !aligned_to(workspace, kAlign))
    return SPEC_ERR_MISALIGNED;
  size_t need = 0;
  spec_greedy_workspace_size(batch, gamma_max, &need);
  if (workspace_bytes < need) return SPEC_ERR_WORKSPACE;
  const GreedyLayout L = greedy_layout(batch, gamma_max);
  char* ws = static_cast<char*>(workspace);
  GreedyArgs a;
  a.early_logits = g_early_logits.load(std::memory_order_relaxed);
  a.tgt = static_cast<const char*>(target_logits);
  a.tokens = draft_tokens;
  a.gammas = gamma_per_seq;
  a.B = batch;
  a.G = gamma_max;
  a.V = vocab;
  a.aligned = (vocab % elems_per_vec(dtype) == 0) && aligned_to(target_logits, 16);
  a.row_bytes = static_cast<size_t>(vocab) * es;
  a.counters = reinterpret_cast<uint32_t*>(ws + L.counters);
  a.rows = reinterpret_cast<int2*>(ws + L.rows);
  a.out_tokens = out_tokens;
  a.out_nacc = out_num_accepted;
  a.out_status = out_status;
  uint32_t* stop_enc = reinterpret_cast<uint32_t*>(ws + L.stop);
  const unsigned grid = static_cast<unsigned>(batch) * static_cast<unsigned>(gamma_max + 1);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (dtype == SPEC_BF16) {
    err = prepare(greedy_early_kernel<DT_BF16>, g_ready[8]);
    if (err == cudaSuccess)
      greedy_early_kernel<DT_BF16><<<grid, kThreads, sizeof(Smem), s>>>(a, stop_enc, out_rows_read);
  } else {
    err = prepare(greedy_early_kernel<DT_F32>, g_ready[9]);
    if (err == cudaSuccess)
      greedy_early_kernel<DT_F32><<<grid, kThreads, sizeof(Smem), s>>>(a, stop_enc, out_rows_read);
  }
  if (err == cudaSuccess) err = cudaGetLastError();
  return err == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

spec_status_t spec_transform_probs(const void* logits, spec_dtype_t dtype, int32_t rows, int32_t vocab,
                                   spec_sampling_params_t params, float* out_probs,
                                   int32_t* out_row_status, void* stream) {
  if (dtype != SPEC_BF16 && dtype != SPEC_F32) return SPEC_ERR_INVALID_ARG;
  if (rows < 1 || vocab < 1 || !params_ok(params) || !logits || !out_probs) return SPEC_ERR_INVALID_ARG;
  const size_t es = elem_bytes(dtype);
  if (!aligned_to(logits, es) || !aligned_to(out_probs, 4) || !aligned_to(out_row_status, 4))
    return SPEC_ERR_MISALIGNED;
  const RowParams P = make_row_params(params, vocab, dtype);
  const int aligned = (vocab % elems_per_vec(dtype) == 0) && aligned_to(logits, 16);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const char* lg = static_cast<const char*>(logits);
  const size_t rb = static_cast<size_t>(vocab) * es;
  cudaError_t err;
  if (dtype == SPEC_BF16) {
    err = prepare(transform_kernel<DT_BF16>, g_ready[4]);
    if (err == cudaSuccess)
      transform_kernel<DT_BF16><<<rows, kThreads, smem_for(P, P, SPEC_BF16), s>>>(lg, vocab, P, aligned, rb, out_probs,
                                                                               out_row_status);
  } else {
    err = prepare(transform_kernel<DT_F32>, g_ready[5]);
    if (err == cudaSuccess)
      transform_kernel<DT_F32><<<rows, kThreads, smem_for(P, P, SPEC_F32), s>>>(lg, vocab, P, aligned, rb, out_probs,
                                                                             out_row_status);
  }
  if (err == cudaSuccess) err = cudaGetLastError();
  return err == cudaSuccess ? SPEC_OK : SPEC_ERR_CUDA;
}

}  // extern "C"

// Five row CTAs must fit on one SM (228 KB of shared memory, 1 KB reserved per CTA).
static_assert(5 * (sizeof(sv::Smem) + 1024) <= 228 * 1024, "row CTA shared memory too large for 5 CTAs per SM");

// ====================================================================== allocation-free variant
// Scratch for spec_verify_sample_noalloc: a fixed-size array in the library's
// own device memory, present on every GPU that loads the library until the
// process exits.  All calls share it.
namespace {

constexpr size_t kStaticScratchBytes = 8u << 20;   // 8 MiB
static __device__ __align__(256) unsigned char g_static_scratch[kStaticScratchBytes];

// Device address of g_static_scratch on the current device.  Host code only
// sees a stand-in symbol, never a usable pointer, so the address is asked of
// the runtime: on every call made outside stream capture (a cudaDeviceReset
// reloads the module, and the array may move), and from the per-device cache
// while the stream is being captured (the runtime is not asked then; a first
// call under capture finds no cache and fails with SPEC_ERR_CUDA).
std::atomic<void*> g_scratch_addr[64];

cudaError_t static_scratch(cudaStream_t stream, void** out) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  err = cudaStreamIsCapturing(stream, &cap);
  if (err != cudaSuccess) return err;
  void* p = nullptr;
  if (cap == cudaStreamCaptureStatusNone) {
    err = cudaGetSymbolAddress(&p, g_static_scratch);
    if (err != cudaSuccess) return err;
    g_scratch_addr[dev].store(p, std::memory_order_release);
  } else {
    p = g_scratch_addr[dev].load(std::memory_order_acquire);
    if (p == nullptr) return cudaErrorStreamCaptureUnsupported;
  }
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" SPEC_API spec_status_t spec_verify_sample_noalloc(
    const void* target_logits, const void* draft_logits, spec_dtype_t dtype, const int32_t* draft_tokens,
    const int32_t* gamma_per_seq, const uint8_t* draft_is_onehot, const float* u_accept,
    const float* u_sample, spec_sampling_params_t target_params, spec_sampling_params_t draft_params,
    int32_t batch, int32_t gamma_max, int32_t vocab, int32_t* out_tokens, int32_t* out_num_accepted,
    float* out_accept_prob, float* out_residual_z, int32_t* out_status, void* stream) {
  size_t need = 0;
  const spec_status_t st = spec_verify_workspace_size(batch, gamma_max, vocab, target_params,
                                                      draft_params, &need);
  if (st != SPEC_OK) return st;
  if (need > kStaticScratchBytes) return SPEC_ERR_WORKSPACE;   // beyond the 8 MiB static scratch
  void* scratch = nullptr;
  if (static_scratch(static_cast<cudaStream_t>(stream), &scratch) != cudaSuccess) return SPEC_ERR_CUDA;
  // The per-sequence counters at the start of the scratch must be zero when the
  // kernels start: verify_sample_impl clears them on the caller's stream once
  // every host check has passed (an invalid call launches nothing and leaves
  // the scratch as it was).
  return verify_sample_impl(target_logits, draft_logits, dtype, draft_tokens, gamma_per_seq,
                            draft_is_onehot, u_accept, u_sample, target_params, draft_params, nullptr,
                            batch, gamma_max, vocab, scratch, kStaticScratchBytes, out_tokens,
                            out_num_accepted, out_accept_prob, out_residual_z, out_status, nullptr, stream,
                            true);
}
