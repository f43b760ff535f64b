// sv_row.cuh -- per-row analysis of one logits row by one CTA (sm_103a).
//
// A row is the logits vector z over the vocabulary for one (sequence,
// position) of the target or the draft.  The analysis produces what the
// verifier needs from that row [wrblog §7.2, §7.3]:
//   * the row maximum m and the normaliser W of the kept set,
//   * the kept set itself (a compact list when top-k is small, otherwise a
//     threshold "composite >= cut" on the ordering of sv_common.cuh),
//   * the probability of the one draft token this row scores,
//   * a status (NaN / +inf logits, or a row of only -inf).
//
// Two algorithms:
//   PATH_STREAM (1 <= top_k <= kSmallK): one streaming pass from HBM.  Each
//     warp keeps a threshold filter: an element enters the warp's candidate
//     buffer only if it beats the k-th largest element the warp has kept so
//     far; when the buffer fills, a warp radix select re-establishes the
//     top-k.  The block then merges the warps' top-k, sorts the k survivors
//     and evaluates softmax and the top-p cut over them in float64.
//   PATH_FULL (top_k off or large): pass 1 streams the row once for the
//     maximum (and, with no cut at all, the softmax denominator: per-thread
//     online rescaling, Kahan-compensated float sums, float64 across
//     threads).  A large top-k is found by MSB-first radix selection over
//     re-reads of the row (digit histograms of counts); a top-p cut by
//     bracketing (see "PATH_FULL top-p by bracketing" below), with radix
//     selection over exact 64-bit fixed-point masses as its fallback.
//
// Sources: [wrblog] "推测解码：草稿模型、接受率、正确性与加速边界" (wrblog.cn).
#pragma once

#include "sv_common.cuh"

namespace sv {

static_assert(kThreads >= 256 && kThreads % 32 == 0, "block-wide 256-bin histograms assume at least 256 threads");

struct RowParams {
  float T;          // temperature (> 0)
  float cT;         // log2(e) / T as float: 2^((z - m) * cT) = exp((z - m) / T)
  float cT_lo;      // log2(e) / T - cT (the float rounding error of cT)
  double invT;      // 1 / T in float64
  int k;            // top-k, 0 = off (the host maps k >= V to 0)
  float top_p;      // 1 = off
  int path;         // PATH_STREAM or PATH_FULL
  int fixed_shift;  // fixed-point scale 2^fixed_shift for probability masses
  int lazy;         // PATH_FULL top-p: leave open which ties of the cut value come first (RowStat::n_list)
};

// Per-row result, mirrored into the workspace for the sequence epilogue.
struct __align__(16) RowStat {
  double W;        // PATH_FULL: normaliser, sum over the kept set of exp((z - m) / T)
  uint64_t cut;    // PATH_FULL: token kept iff composite >= cut (0 keeps all)
  float m;         // row maximum
  float p_tok;     // probability of the draft token this row scores (0 if none)
  int32_t status;  // SEQ_OK, SEQ_NONFINITE or SEQ_EMPTY_SUPPORT
  int32_t n_list;  // PATH_STREAM: kept-list length.  PATH_FULL: 0, or n > 0 when the row left
                   // open which of its elements equal to the cut value come first: cut then
                   // counts every such tie as kept, and only the first n of them in index
                   // order are (the full-row draw resolves them by rank)
  int32_t path;
  int32_t argmax;  // greedy rows: argmax token
  float cT;        // the row's log2(e) / T (its sampling rule, for the draw)
  float invW;      // PATH_FULL: (float)(1 / W), formed once per row (float64 is slow here)
};
static_assert(sizeof(RowStat) == 48, "RowStat layout");

struct __align__(16) ListEntry {  // one kept token of a PATH_STREAM row
  float p, p_lo;                  // its probability as a double-float (hi, lo)
  int32_t token;
  int32_t pad;
};

// ------------------------------------------------------------------ shared memory
struct __align__(16) SmemFull {
  unsigned long long mass[256];
  unsigned long long mx[256];
  uint32_t cnt[256];
  uint32_t wcnt[kWarps];
};
struct __align__(16) SmemEpi {
  int32_t tok[kListCap];             // list draw: the target kept list's tokens
  int32_t qtok[kListCap];            // draft kept list (token order, for lookups)
  float qp[kListCap];
  float wh[kWarps], wl[kWarps];      // list draw: per-warp scan totals, double-float
  double wtot[kWarps];               // per-warp segment totals of the block scan
  double csum[kWarps][kScanChunks];  // per-chunk totals of the block scan
  RowStat rs[2 * kMaxGamma + 1];     // the sequence's row summaries
};
struct __align__(16) Smem {
  union {
    SmemFull f;
    SmemEpi e;
    uint4 ring[kRing][kThreads];     // PATH_STREAM pass 1: each thread's cp.async ring of vectors
  } u;
  uint32_t khist[2][256];            // PATH_STREAM: digit histograms of the per-thread maxima
  alignas(16) uint64_t cand[kCandCap];   // PATH_STREAM: candidates (composites >= the lower bound)
  alignas(16) uint64_t topk[kSmallK];
  uint64_t sorted[kSmallK];          // PATH_STREAM: top-k in descending order
  alignas(16) int32_t list_tok[kListCap];   // padded with INT_MAX to a multiple of 4 entries
  float list_ph[kListCap], list_pl[kListCap];   // kept probabilities, double-float
  int nw[kWarps];
  int ncand;
  int nfull;                         // PATH_STREAM: threads whose vectors need a full re-read
  int16_t full[kMaxFull];
  float red_f[kWarps];
  float red_lo[kWarps];
  double red_d[kWarps];
  uint64_t red_u[kWarps];
  int red_i[kWarps];
  int flag_bad;
  // broadcast slots
  uint64_t b_u64[4];
  double b_f64[4];
  float b_f32[2];
  int b_i32[10];
  RowParams rowp;                    // a row's sampling rule when it is given per sequence
  RowStat st;
  // the sequence's draft tokens and uniforms, copied in while the row streams
  // (read by the sequence epilogue)
  int32_t seq_tok[kMaxGamma];
  float seq_u[kMaxGamma];
  float seq_us;
  int early_skip;                    // early exit: this CTA's row is not read
};

// ------------------------------------------------------------------ early-exit stop marks
// A row CTA under early exit watches its sequence's stop mark: once *p > thr
// an earlier position has stopped the sequence, the row's result is never
// used, and the row may be abandoned.  p == nullptr: nothing to watch.
struct StopCheck {
  const unsigned* p = nullptr;
  unsigned thr = 0;
};
__device__ __forceinline__ unsigned ld_relaxed_u32(const unsigned* p) {
  unsigned v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Block-wide (every thread calls it): true when the mark says stop.
__device__ __forceinline__ bool stop_now(const StopCheck& sc, Smem& sm) {
  if (!sc.p) return false;
  __syncthreads();                                 // earlier readers of sm.early_skip are done
  if (threadIdx.x == 0) sm.early_skip = ld_relaxed_u32(sc.p) > sc.thr ? 1 : 0;
  __syncthreads();
  return sm.early_skip != 0;
}
// The summary of an abandoned row (never read by the epilogue).
__device__ __forceinline__ void abandon_row(Smem& sm, float cT) {
  if (threadIdx.x == 0) {
    RowStat st;
    st.W = 1.0; st.cut = 0; st.m = 0.0f; st.p_tok = 0.0f; st.status = SEQ_OK; st.n_list = 0;
    st.path = PATH_FULL; st.argmax = -1; st.cT = cT; st.invW = 0.0f;
    sm.st = st;
  }
  __syncthreads();
}

// ------------------------------------------------------------------ digit walks
// Warp-wide: positions 0..255 visit digits in the order given by `desc`
// (descending digits 255..0, or ascending 0..255).  Finds the position whose
// cumulative count first reaches `need` (1-based rank); returns the digit and
// the count of all earlier positions.
__device__ __forceinline__ void pick_digit_count(const uint32_t* hist, uint32_t need, bool desc,
                                                 int lane, int& digit, uint32_t& before) {
  uint32_t c[8];
  uint32_t s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int pos = 8 * lane + j;
    c[j] = hist[desc ? 255 - pos : pos];
    s += c[j];
  }
  const uint32_t incl = warp_incl_scan_u32(s, lane);
  const uint32_t excl = incl - s;
  const unsigned bal = __ballot_sync(kFull, excl < need && need <= incl);
  const int L = bal ? __ffs(bal) - 1 : 31;
  int d = desc ? 0 : 255;
  uint32_t bf = excl;
  if (lane == L) {
    uint32_t acc = excl;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int pos = 8 * lane + j;
      if (acc + c[j] >= need) { d = desc ? 255 - pos : pos; bf = acc; break; }
      acc += c[j];
    }
  }
  digit = __shfl_sync(kFull, d, L);
  before = __shfl_sync(kFull, bf, L);
}

// Mass version: first position where before + mass >= tau (64-bit exact).
__device__ __forceinline__ void pick_digit_mass(const unsigned long long* mass, uint64_t base,
                                                uint64_t tau, bool desc, int lane, int& digit,
                                                uint64_t& before) {
  uint64_t c[8];
  uint64_t s = 0;
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const int pos = 8 * lane + j;
    c[j] = mass[desc ? 255 - pos : pos];
    s += c[j];
  }
  uint64_t incl = s;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint64_t t = shfl_u64(incl, (lane - o) & 31);
    if (lane >= o) incl += t;
  }
  const uint64_t excl = incl - s;
  const unsigned bal = __ballot_sync(kFull, base + excl < tau && tau <= base + incl);
  // If rounding left the total short of tau, take the last non-empty position.
  int L = bal ? __ffs(bal) - 1 : -1;
  if (L < 0) {
    const unsigned nz = __ballot_sync(kFull, s != 0);
    L = nz ? 31 - __clz(nz) : 31;
  }
  int d = desc ? 0 : 255;
  uint64_t bf = excl;
  if (lane == L) {
    uint64_t acc = excl;
    int last_nz = -1;
    uint64_t acc_last = excl;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int pos = 8 * lane + j;
      if (c[j] != 0) { last_nz = pos; acc_last = acc; }
      if (base + acc + c[j] >= tau && c[j] != 0) { d = desc ? 255 - pos : pos; bf = acc; last_nz = -2; break; }
      acc += c[j];
    }
    if (last_nz >= 0) { d = desc ? 255 - last_nz : last_nz; bf = acc_last; }
  }
  digit = __shfl_sync(kFull, d, L);
  before = shfl_u64(bf, L);
}

// ------------------------------------------------------------------ block reductions
__device__ __forceinline__ float block_max_f(float v, Smem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
  if (lane == 0) sm.red_f[warp] = v;
  __syncthreads();
  float r = sm.red_f[0];
  for (int w = 1; w < kWarps; ++w) r = fmaxf(r, sm.red_f[w]);
  __syncthreads();
  return r;
}
__device__ __forceinline__ double block_sum_d(double v, Smem& sm) {
  // float64 adds are slow on this part: one thread adds the warps' partials
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_f64(v);
  if (lane == 0) sm.red_d[warp] = v;
  __syncthreads();
  if (threadIdx.x == 0) {
    double r = 0.0;
    for (int w = 0; w < kWarps; ++w) r += sm.red_d[w];
    sm.b_f64[3] = r;
  }
  __syncthreads();
  const double r = sm.b_f64[3];
  __syncthreads();
  return r;
}
// A block sum of float terms in double-float (float pipe only), returned as a double.
__device__ __forceinline__ double block_sum_fd(float v, Smem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const df w = warp_sum_df(df_from(v));
  if (lane == 0) {
    sm.red_f[warp] = w.hi;
    sm.red_lo[warp] = w.lo;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    df r = df_from(0.0f);
    for (int k = 0; k < kWarps; ++k) r = df_add(r, {sm.red_f[k], sm.red_lo[k]});
    sm.b_f64[3] = df_to_double(r);
  }
  __syncthreads();
  const double r = sm.b_f64[3];
  __syncthreads();
  return r;
}
__device__ __forceinline__ int block_or(int v, Smem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = __any_sync(kFull, v) ? 1 : 0;
  if (lane == 0) sm.red_i[warp] = v;
  __syncthreads();
  int r = 0;
  for (int w = 0; w < kWarps; ++w) r |= sm.red_i[w];
  __syncthreads();
  return r;
}
__device__ __forceinline__ uint64_t block_max_u64(uint64_t v, Smem& sm) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max_u64(v);
  if (lane == 0) sm.red_u[warp] = v;
  __syncthreads();
  uint64_t r = 0;
  for (int w = 0; w < kWarps; ++w) r = sm.red_u[w] > r ? sm.red_u[w] : r;
  __syncthreads();
  return r;
}

// ------------------------------------------------------------------ greedy row
// argmax_x z(x), lowest index on ties [wrblog §7.1]; status for NaN / +inf / all -inf.
// sc: the early-exit stop mark to watch (none by default); a warp that sees
// it set stops reading and raises sm.early_skip, which the caller has cleared
// behind a barrier and reads after this function returns.
template <int DT>
__device__ void greedy_row(const Row row, Smem& sm, int& argmax, int& status, const StopCheck sc = StopCheck()) {
  constexpr int P = Elem<DT>::kPer;
  const int tid = threadIdx.x;
  float best = -__int_as_float(0x7f800000);
  int best_i = -1;
  bool bad = false;
  unsigned seen = 0u;     // the stop mark as read two iterations earlier (one load per warp)
  int it = 0;
  for (int base = 0; base < row.nvec; base += kThreads * kUnroll, ++it) {
    if (sc.p && (it & 1)) {
      if (seen > sc.thr) {                             // the sequence stopped: abandon the row
        if ((tid & 31) == 0) sm.early_skip = 1;
        break;
      }
      seen = ld_relaxed_u32(sc.p);                     // consumed two iterations later
    }
    uint4 r[kUnroll];
    int cnt[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) cnt[u] = load_vec<DT, true>(row, base + u * kThreads + tid, r[u]);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (cnt[u] == 0) continue;
      bool vb;
      const float vm = vec_max<DT>(r[u], cnt[u], vb);
      bad |= vb;
      if (vm > best) {           // strictly greater: earlier (lower) indices win ties
        float x[P];
        unpack<DT>(r[u], x);
        int e = 0;
#pragma unroll
        for (int j = P - 1; j >= 0; --j)
          if (j < cnt[u] && x[j] == vm) e = j;
        best = vm;
        best_i = (base + u * kThreads + tid) * P + e;
      }
    }
  }
  const uint64_t c = best_i >= 0 ? composite(fkey(best), static_cast<uint32_t>(best_i)) : 0ull;
  const uint64_t top = block_max_u64(c, sm);
  const int any_bad = block_or(bad ? 1 : 0, sm);
  status = any_bad ? SEQ_NONFINITE : (top == 0ull ? SEQ_EMPTY_SUPPORT : SEQ_OK);
  argmax = top == 0ull ? -1 : static_cast<int>(comp_index(top));
}

// ------------------------------------------------------------------ PATH_FULL
// Fixed-point mass of a weight w in [0, 1].
__device__ __forceinline__ unsigned long long fixed_mass(float w, float scale) {
  return __float2ull_rn(w * scale);
}
// Log-probability bucket: eight buckets per factor of two below the maximum.
__device__ __forceinline__ int tbin_of(float t) {
  const float f = fminf(-t * 8.0f, 255.0f);
  return static_cast<int>(f);
}

// Pass 1: maximum and softmax denominator of the whole row.
template <int DT>
__device__ void full_pass1(const Row row, float cT, Smem& sm, float& m_out, double& S_out, int& bad_out) {
  constexpr int P = Elem<DT>::kPer;
  const int tid = threadIdx.x;
  const float NEG_INF = -__int_as_float(0x7f800000);
  float m = NEG_INF, s = 0.0f, comp = 0.0f;
  bool bad = false;
  for (int base = 0; base < row.nvec; base += kThreads * kUnroll) {
    uint4 r[kUnroll];
    int cnt[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) cnt[u] = load_vec<DT, false>(row, base + u * kThreads + tid, r[u]);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (cnt[u] == 0) continue;
      bool vb;
      const float vm = vec_max<DT>(r[u], cnt[u], vb);
      bad |= vb;
      if (vm > m) {
        if (m > NEG_INF) {
          const float f = fast_exp2((m - vm) * cT);
          s *= f;
          comp *= f;
        }
        m = vm;
      }
      if (m > NEG_INF) {
        float x[P];
        unpack<DT>(r[u], x);
        float vs = 0.0f;
#pragma unroll
        for (int e = 0; e < P; ++e)
          if (e < cnt[u]) vs += fast_exp2((x[e] - m) * cT);
        const float y = vs - comp;           // Kahan-compensated accumulation
        const float t = s + y;
        comp = (t - s) - y;
        s = t;
      }
    }
  }
  const float mb = block_max_f(m, sm);
  double term = 0.0;
  if (m > NEG_INF && mb > NEG_INF) term = static_cast<double>(s) * static_cast<double>(fast_exp2((m - mb) * cT));
  const double S = block_sum_d(term, sm);
  bad_out = block_or(bad ? 1 : 0, sm);
  m_out = mb;
  S_out = S;
}

// Sum over the kept set {composite >= cut} of 2^((z - m) cT), float64 across threads.
template <int DT>
__device__ __noinline__ double full_sum_kept(const Row row, float m, float cT, uint64_t cut, Smem& sm) {
  constexpr int P = Elem<DT>::kPer;
  const int tid = threadIdx.x;
  float s = 0.0f, comp = 0.0f;
  for (int base = 0; base < row.nvec; base += kThreads * kUnroll) {
    uint4 r[kUnroll];
    int cnt[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) cnt[u] = load_vec<DT, false>(row, base + u * kThreads + tid, r[u]);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (cnt[u] == 0) continue;
      float x[P];
      unpack<DT>(r[u], x);
      const int v = base + u * kThreads + tid;
      float vs = 0.0f;
#pragma unroll
      for (int e = 0; e < P; ++e) {
        if (e < cnt[u] && composite(fkey(x[e]), static_cast<uint32_t>(v * P + e)) >= cut)
          vs += fast_exp2((x[e] - m) * cT);
      }
      const float y = vs - comp;
      const float t = s + y;
      comp = (t - s) - y;
      s = t;
    }
  }
  return block_sum_fd(s, sm);
}

// Warp segments: warp w owns the contiguous vectors [w L, (w + 1) L) of a row,
// so counts per warp are counts per index range.
__device__ __forceinline__ int seg_len(const Row row) { return (row.nvec + kWarps - 1) / kWarps; }

// Raw element bits that carry order key K: the value's own bits and, for a
// zero, those of -0 as well (keys fold -0 onto +0).
template <int DT>
struct KeyBits {
  uint32_t a, b;
  __device__ __forceinline__ explicit KeyBits(uint32_t K) {
    const uint32_t v = __float_as_uint(key_value(K));
    a = DT == DT_BF16 ? (v >> 16) : v;
    b = (v & 0x7fffffffu) == 0u ? (DT == DT_BF16 ? 0x8000u : 0x80000000u) : a;
  }
  __device__ __forceinline__ bool hit(uint32_t x) const { return x == a || x == b; }
  // Elements e < c of vector q that carry the key, as a bit mask.
  __device__ __forceinline__ uint32_t mask(const uint4& q, int c) const {
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
    uint32_t m = 0;
#pragma unroll
    for (int e = 0; e < Elem<DT>::kPer; ++e) {
      const uint32_t x = DT == DT_BF16 ? ((e & 1) ? (w[e >> 1] >> 16) : (w[e >> 1] & 0xffffu)) : w[e];
      m |= (e < c && hit(x)) ? (1u << e) : 0u;
    }
    return m;
  }
};

// Index of the r-th (1-based) element with key K in vectors [v0, v1), in
// index order; -1 if there are fewer.  Block-wide: while the range is long,
// every warp counts K in one eighth of it (kUnroll loads in flight per lane)
// and the range shrinks to the eighth holding the r-th; one warp then scans.
template <int DT>
__device__ __noinline__ int range_find_nth(const Row row, uint32_t K, int v0, int v1, uint32_t r, Smem& sm) {
  constexpr int P = Elem<DT>::kPer;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const KeyBits<DT> kb(K);
  while (v1 - v0 > 32 * kWarps) {
    const int sub = (v1 - v0 + kWarps - 1) / kWarps;
    const int a0 = v0 + warp * sub, a1 = min(v1, a0 + sub);
    uint32_t my = 0;
    for (int s = a0; s < a1; s += 32 * kUnroll) {
      uint4 q[kUnroll];
      int c[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int v = s + u * 32 + lane;
        c[u] = v < a1 ? load_vec<DT, false>(row, v, q[u]) : 0;
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) my += __popc(kb.mask(q[u], c[u]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) my += __shfl_xor_sync(kFull, my, o);
    if (lane == 0) sm.u.f.wcnt[warp] = my;
    __syncthreads();
    if (tid == 0) {
      uint32_t acc = 0;
      int W = -1;
      for (int w = 0; w < kWarps; ++w) {
        if (acc + sm.u.f.wcnt[w] >= r) { W = w; break; }
        acc += sm.u.f.wcnt[w];
      }
      sm.b_i32[4] = W;
      sm.b_i32[5] = static_cast<int>(r - acc);
    }
    __syncthreads();
    const int W = sm.b_i32[4];
    r = static_cast<uint32_t>(sm.b_i32[5]);
    __syncthreads();
    if (W < 0) return -1;                   // same in every thread
    v0 = v0 + W * sub;
    v1 = min(v1, v0 + sub);
  }
  if (tid == 0) sm.b_i32[6] = -1;
  __syncthreads();
  if (warp == 0) {
    uint32_t running = 0;
    for (int s = v0; s < v1; s += 32) {
      const int v = s + lane;
      uint4 q;
      const int c = v < v1 ? load_vec<DT, false>(row, v, q) : 0;
      const uint32_t hits = kb.mask(q, c);
      const uint32_t mine = __popc(hits);
      const uint32_t incl = warp_incl_scan_u32(mine, lane);
      const unsigned bal = __ballot_sync(kFull, running + incl >= r && mine > 0);
      if (bal) {
        const int Lw = __ffs(bal) - 1;
        if (lane == Lw) {
          // the (r - before)-th set bit of this lane's hit mask
          uint32_t h = hits;
          for (uint32_t k = running + incl - mine + 1; k < r; ++k) h &= h - 1;
          sm.b_i32[6] = v * P + (__ffs(h) - 1);
        }
        break;
      }
      running += __shfl_sync(kFull, incl, 31);
    }
  }
  __syncthreads();
  return sm.b_i32[6];
}

// Index of the n-th (1-based) element, in index order, whose key equals K.
template <int DT>
__device__ __forceinline__ int find_nth_with_key(const Row row, uint32_t K, uint32_t n, Smem& sm) {
  return range_find_nth<DT>(row, K, 0, row.nvec, n, sm);
}

// Elements with key K among indices [0, x), block-wide (the same in every thread).
template <int DT>
__device__ __noinline__ uint32_t count_key_before(const Row row, uint32_t K, int x, Smem& sm) {
  constexpr int P = Elem<DT>::kPer;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const KeyBits<DT> kb(K);
  const int vfull = x / P;                    // vectors wholly before x
  uint32_t my = 0;
  for (int s = 0; s < vfull; s += kThreads * kUnroll) {
    uint4 q[kUnroll];
    int c[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = s + u * kThreads + tid;
      c[u] = v < vfull ? load_vec<DT, false>(row, v, q[u]) : 0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) my += __popc(kb.mask(q[u], c[u]));
  }
  if (tid == 0 && x % P) {
    uint4 q;
    const int c = load_vec<DT, false>(row, vfull, q);
    my += __popc(kb.mask(q, min(c, x % P)));
  }
  my = __reduce_add_sync(kFull, my);
  if (lane == 0) sm.u.f.wcnt[warp] = my;
  __syncthreads();
  uint32_t tot = 0;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) tot += sm.u.f.wcnt[w];
  __syncthreads();
  return tot;
}

// One radix round over a re-read of the row.  Elements taking part: composite
// >= ck, and (if tb >= 0) in log-probability bucket tb, and matching prefix
// under mask.  kind 0: digit = bucket of log-probability; kind 1: digit = the
// composite byte at `shift`.  Accumulates counts, fixed-point masses (when
// with_mass) and the largest composite per digit.
template <int DT>
__device__ __noinline__ void full_round(const Row row, float m, float cT, float scale, uint64_t ck, int tb,
                           uint64_t prefix, uint64_t mask, int kind, int shift, bool with_mass,
                           Smem& sm) {
  constexpr int P = Elem<DT>::kPer;
  const int tid = threadIdx.x;
  if (tid < 256) {
    sm.u.f.cnt[tid] = 0u;
    sm.u.f.mass[tid] = 0ull;
    sm.u.f.mx[tid] = 0ull;
  }
  __syncthreads();
  for (int base = 0; base < row.nvec; base += kThreads * kUnroll) {
    uint4 r[kUnroll];
    int cnt[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) cnt[u] = load_vec<DT, false>(row, base + u * kThreads + tid, r[u]);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (cnt[u] == 0) continue;
      float x[P];
      unpack<DT>(r[u], x);
      const int v = base + u * kThreads + tid;
#pragma unroll
      for (int e = 0; e < P; ++e) {
        if (e >= cnt[u]) continue;
        const uint64_t c = composite(fkey(x[e]), static_cast<uint32_t>(v * P + e));
        if (c < ck) continue;
        const float t = (x[e] - m) * cT;
        if (tb >= 0 && tbin_of(t) != tb) continue;
        if ((c & mask) != prefix) continue;
        const int d = kind == 0 ? tbin_of(t) : static_cast<int>((c >> shift) & 255u);
        atomicAdd(&sm.u.f.cnt[d], 1u);
        atomicMax(&sm.u.f.mx[d], static_cast<unsigned long long>(c));
        if (with_mass) atomicAdd(&sm.u.f.mass[d], fixed_mass(fast_exp2(t), scale));
      }
    }
  }
  __syncthreads();
}

// k-th largest composite of the row (count-based radix select).
template <int DT>
__device__ __noinline__ uint64_t full_select_topk(const Row row, float m, float cT, int k, Smem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t prefix = 0, mask = 0;
  uint32_t need = static_cast<uint32_t>(k);
  const int last_shift = DT == DT_BF16 ? 48 : 32;
  for (int shift = 56; shift >= last_shift; shift -= 8) {
    full_round<DT>(row, m, cT, 1.0f, 0ull, -1, prefix, mask, 1, shift, false, sm);
    if (warp == 0) {
      int digit;
      uint32_t before;
      pick_digit_count(sm.u.f.cnt, need, true, lane, digit, before);
      if (lane == 0) {
        sm.b_i32[0] = digit;
        sm.b_i32[1] = static_cast<int>(before);
        sm.b_i32[2] = static_cast<int>(sm.u.f.cnt[digit]);
        sm.b_u64[1] = sm.u.f.mx[digit];
      }
    }
    __syncthreads();
    const int digit = sm.b_i32[0];
    need -= static_cast<uint32_t>(sm.b_i32[1]);
    const int cd = sm.b_i32[2];
    const uint64_t mx = sm.b_u64[1];
    prefix |= static_cast<uint64_t>(digit) << shift;
    mask |= 0xffull << shift;
    __syncthreads();
    if (cd == 1) return mx;
    if (shift == last_shift) {
      const uint32_t K = static_cast<uint32_t>(mx >> 32);   // every element left has this key
      const int idx = find_nth_with_key<DT>(row, K, need, sm);
      return composite(K, static_cast<uint32_t>(idx));
    }
  }
  return prefix;
}

// Top-p cut among {composite >= ck}: the largest composite c* whose inclusive
// cumulative mass (descending order) reaches top_p of the kept mass.  Returns
// c* and the fixed-point kept mass through c*.
template <int DT>
__device__ __noinline__ uint64_t full_select_topp(const Row row, float m, float cT, float scale, uint64_t ck,
                                     float top_p, Smem& sm, unsigned long long& Wfixed) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // round 0: log-probability buckets, ascending = descending probability
  full_round<DT>(row, m, cT, scale, ck, -1, 0ull, 0ull, 0, 0, true, sm);
  if (warp == 0) {
    uint64_t tot = 0;
    for (int j = lane; j < 256; j += 32) tot += sm.u.f.mass[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += shfl_xor_u64(tot, o);
    double tf = ceil(static_cast<double>(top_p) * static_cast<double>(tot));
    uint64_t tau = tf >= static_cast<double>(tot) ? tot : static_cast<uint64_t>(tf);
    if (tau == 0) tau = 1;
    int digit;
    uint64_t before;
    pick_digit_mass(sm.u.f.mass, 0ull, tau, false, lane, digit, before);
    if (lane == 0) {
      sm.b_u64[0] = tau;
      sm.b_u64[1] = before;
      sm.b_u64[2] = sm.u.f.mx[digit];
      sm.b_u64[3] = sm.u.f.mass[digit];
      sm.b_i32[0] = digit;
      sm.b_i32[2] = static_cast<int>(sm.u.f.cnt[digit]);
    }
  }
  __syncthreads();
  const uint64_t tau = sm.b_u64[0];
  uint64_t above = sm.b_u64[1];
  const int tb = sm.b_i32[0];
  int cd = sm.b_i32[2];
  uint64_t mx = sm.b_u64[2];
  uint64_t md = sm.b_u64[3];
  __syncthreads();
  if (cd == 1) { Wfixed = above + md; return mx; }

  uint64_t prefix = 0, mask = 0;
  const int last_shift = DT == DT_BF16 ? 48 : 32;
  for (int shift = 56; shift >= last_shift; shift -= 8) {
    full_round<DT>(row, m, cT, scale, ck, tb, prefix, mask, 1, shift, true, sm);
    if (warp == 0) {
      int digit;
      uint64_t before;
      pick_digit_mass(sm.u.f.mass, above, tau, true, lane, digit, before);
      if (lane == 0) {
        sm.b_u64[1] = before;
        sm.b_u64[2] = sm.u.f.mx[digit];
        sm.b_u64[3] = sm.u.f.mass[digit];
        sm.b_i32[0] = digit;
        sm.b_i32[2] = static_cast<int>(sm.u.f.cnt[digit]);
      }
    }
    __syncthreads();
    const int digit = sm.b_i32[0];
    above += sm.b_u64[1];
    mx = sm.b_u64[2];
    md = sm.b_u64[3];
    cd = sm.b_i32[2];
    prefix |= static_cast<uint64_t>(digit) << shift;
    mask |= 0xffull << shift;
    __syncthreads();
    if (cd == 1) { Wfixed = above + md; return mx; }
  }
  // every remaining element has the same key, hence the same mass
  const uint32_t K = static_cast<uint32_t>(mx >> 32);
  const uint64_t wf = md / static_cast<uint64_t>(cd);
  uint64_t nneed = (wf && tau > above) ? (tau - above + wf - 1) / wf : 1;
  if (nneed < 1) nneed = 1;
  if (nneed > static_cast<uint64_t>(cd)) nneed = cd;
  const int idx = find_nth_with_key<DT>(row, K, static_cast<uint32_t>(nneed), sm);
  Wfixed = above + nneed * wf;
  return composite(K, static_cast<uint32_t>(idx));
}

// ------------------------------------------------------------------ PATH_FULL top-p by bracketing
// The top-p cut of a full row without radix rounds.  An element's mass
// depends on its value only, so masses can be counted per distinct key:
//   1. bucket pass: the kept masses summed per log-probability class -- kNB
//      buckets of one width below a level top, plus one class above and one
//      below -- in per-thread private float columns of shared memory (no
//      atomics, no bank conflicts).  The class where the cumulative mass
//      (largest first) reaches top_p, widened to its neighbours when the float
//      sums leave the crossing within a margin of a class edge, is the bracket.
//   2. exact pass: the masses above and below the bracket are summed per
//      thread (Kahan float; float64 across threads), and every element inside
//      the bracket is counted per distinct key in a small hash table, one
//      count per warp segment.  A key's mass is its count times its weight.
//   3. resolve: the bracket's keys in descending order give the crossing key
//      K*, how many of its ties the prefix takes, and W; the per-warp counts
//      name the warp segment holding the last tie taken, and one warp scans
//      that eighth of the row for its index.
// A bracket holding more distinct keys than the table is refined by another
// bucket pass over its own range (float32 rows, whose values rarely repeat,
// need this); after kMaxLevels levels the radix rounds above take over.
constexpr int kNB = 32;                 // buckets per level
constexpr int kNC = kNB + 2;            // classes: above, kNB buckets, below
constexpr float kLevel0Width = 1.5f;    // log2 units; level 0 spans 48 below the maximum
constexpr int kNTBits = 8;
constexpr int kNT = 1 << kNTBits;       // bracket key table slots (one per thread)
constexpr int kProbe = 8;               // linear probes before a key counts as overflow
constexpr int kMaxLevels = 3;
constexpr uint32_t kNoKey = 0xffffffffu;  // the key of a NaN: never a key of a finite row
static_assert(kNT == kThreads, "one table slot per thread");

// ------------------------------------------------------------------ PATH_FULL top-p by key counts (bf16)
// A bf16 row has at most 65536 distinct values and usually a few hundred to
// a few thousand; an element's probability depends on its value alone.  So
// the streaming pass that takes the maximum also counts the elements per
// distinct value, with no exponential per element:
//   * values with |z| in [2^-3, 2^5) -- the bulk of a logits row -- index a
//     direct table by (sign, binade, 7 mantissa bits): one red.shared per
//     element, no key check;
//   * any other value goes to a small open-addressing table keyed by its
//     16-bit order key; -inf is skipped (probability 0).
// Counts are kept per half of the row (warps 0-3 and 4-7 each stream their
// own half; two tables count as fast as four and leave room for four CTAs
// per SM instead of three).  The cut then follows from the tables:
//   * per value: weight 2^((z - m) cT) as a 64-bit fixed-point mass, times
//     its count, summed into 256 log-probability bins (exact integer sums);
//   * the bin where the cumulative mass (largest first) reaches
//     ceil(top_p x total) -- the same tau as the radix rounds -- and, inside
//     it, the values in descending order give the crossing value K* and how
//     many of its ties the prefix takes;
//   * for a row that needs it (an exact cut), the per-half counts of K* name
//     the half holding the last tie taken, and a hierarchical count over that
//     half finds its index; a lazy cut leaves it to the draw.
// An overflow of the small table (too many distinct values outside the
// window) hands the row to bracketing, which reuses the maximum (or, in a
// launch given only the count tables' memory, to the radix rounds).
constexpr int kKCDirect = 2048;         // 2 signs x 8 binades x 128 mantissas
constexpr int kKCExpLo = 124;           // biased exponent of 2^-3
constexpr int kKHBits = 8;
constexpr int kKH = 1 << kKHBits;       // small table slots
constexpr int kKHProbe = 16;            // linear probes before overflow
constexpr int kKCSlots = kKCDirect + kKH;
constexpr int kKCList = kCandCap / 2;   // values of the crossing bin (unsorted, then sorted, in sm.cand)
constexpr int kCountTables = 2;         // count rows: one per half of the row (warps 0-3, 4-7)
constexpr int kWarpsPerTable = kWarps / kCountTables;
static_assert(kWarps % kCountTables == 0, "each count table serves whole warps");

struct KeyCount {
  uint32_t cnt[kCountTables][kKCSlots]; // direct slots, then small-table slots
  uint32_t keys[kKH];                   // 16-bit order keys of the small table
};

// Extra shared memory of full-row top-p rows, after Smem.  The value counts
// use only its prefix (bi, bd and the count tables), so a launch whose
// full-row rows all take them asks for kKCExtraBytes and fits more CTAs.
struct __align__(16) FullExtra {
  int bi[8];
  double bd[2];
  union {
    float priv[kNC][kThreads];          // bucket pass: column tid is thread tid's
    struct {
      uint32_t keys[kNT];
      uint32_t cnt[kWarps][kNT];        // per warp segment
      uint32_t skey[kNT];               // bracket keys, descending
      uint32_t scnt[kNT];
      float sw[kNT];
      double smass[kNT];
      int16_t sslot[kNT];
    } t;
    KeyCount kc;                        // bf16 key counts
  } u;
  float csum[kNC];
};
constexpr size_t kKCExtraBytes = offsetof(FullExtra, u) + sizeof(KeyCount);

// Bytes of dynamic shared memory this launch was given.
__device__ __forceinline__ unsigned dyn_smem_bytes() {
  unsigned r;
  asm("mov.u32 %0, %%dynamic_smem_size;" : "=r"(r));
  return r;
}

struct Level {
  float top;    // log2-probability at the top of bucket 1
  float inv_w;  // 1 / bucket width
};
// Class of log-probability t: 0 above the level's range, 1..kNB its buckets
// from the top, kNB + 1 below.  Non-increasing in t, and one function for
// every pass, so each class is a contiguous range of keys.
__device__ __forceinline__ int class_of(float t, const Level& L) {
  float f = fmaf(L.top - t, L.inv_w, 1.0f);
  f = fminf(fmaxf(f, 0.0f), static_cast<float>(kNB + 1));
  return __float_as_int(__fadd_rz(f, 8388608.0f)) - 0x4b000000;   // floor(f), f in [0, 2^23)
}

__device__ __forceinline__ void kahan_add(float& s, float& c, float v) {
  const float y = v - c;
  const float t = s + y;
  c = (t - s) - y;
  s = t;
}

// Pass 1: row maximum and the NaN / +inf flag only.
template <int DT>
__device__ void full_max(const Row row, Smem& sm, float& m_out, int& bad_out) {
  const int tid = threadIdx.x;
  float m = -__int_as_float(0x7f800000);
  bool bad = false;
  for (int base = 0; base < row.nvec; base += kThreads * kUnroll) {
    uint4 r[kUnroll];
    int cnt[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) cnt[u] = load_vec<DT, false>(row, base + u * kThreads + tid, r[u]);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (cnt[u] == 0) continue;
      bool vb;
      m = fmaxf(m, vec_max<DT>(r[u], cnt[u], vb));
      bad |= vb;
    }
  }
  m_out = block_max_f(m, sm);
  bad_out = block_or(bad ? 1 : 0, sm);
}

// Step 1: approximate kept mass per class into fx.csum.
template <int DT>
__device__ __noinline__ void topp_bucket_pass(const Row row, float m, float cT, uint64_t ck, Level L,
                                              Smem& sm, FullExtra& fx) {
  constexpr int P = Elem<DT>::kPer;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t col = smem_u32(&fx.u.priv[0][tid]);   // this thread's column, stride kThreads floats
#pragma unroll
  for (int c = 0; c < kNC; ++c) sts_f32(col + c * kThreads * 4, 0.0f);
  for (int base = 0; base < row.nvec; base += kThreads * kUnroll) {
    uint4 r[kUnroll];
    int cnt[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) cnt[u] = load_vec<DT, false>(row, base + u * kThreads + tid, r[u]);
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (cnt[u] == 0) continue;
      float x[P];
      unpack<DT>(r[u], x);
      const int v = base + u * kThreads + tid;
#pragma unroll
      for (int e = 0; e < P; ++e) {
        if (e >= cnt[u]) continue;
        if (ck != 0ull && composite(fkey(x[e]), static_cast<uint32_t>(v * P + e)) < ck) continue;
        const float t = (x[e] - m) * cT;
        const uint32_t a = col + static_cast<uint32_t>(class_of(t, L)) * (kThreads * 4);
        sts_f32(a, lds_f32(a) + fast_exp2(t));
      }
    }
  }
  __syncthreads();
  for (int c = warp; c < kNC; c += kWarps) {
    float s = 0.0f;
#pragma unroll
    for (int q = 0; q < kThreads / 32; ++q) s += fx.u.priv[c][lane + 32 * q];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(kFull, s, o);
    if (lane == 0) fx.csum[c] = s;
  }
  __syncthreads();
}

// Bracket [lo, hi] of classes around the crossing of top_p in the class sums.
// Every thread computes the same answer from the same shared values.
__device__ __forceinline__ void choose_bracket(const float* cs, float top_p, int& lo, int& hi) {
  float tot = 0.0f;
  for (int c = 0; c < kNC; ++c) tot += cs[c];
  const float tau = top_p * tot, eps = 2e-4f * tot;
  float before = 0.0f;
  int c = 0;
  for (; c < kNC - 1; ++c) {
    if (before + cs[c] >= tau) break;
    before += cs[c];
  }
  lo = hi = c;
  float b_lo = before;                      // approximate mass above class lo
  while (lo > 0 && b_lo >= tau - eps) { --lo; b_lo -= cs[lo]; }
  float a_hi = before + cs[c];              // approximate mass through class hi
  while (hi < kNC - 1 && a_hi < tau + eps) { ++hi; a_hi += cs[hi]; }
}

// Counts key K in the bracket table (per-warp count row cntw); false when the
// probe sequence is full of other keys.
// keys: shared address of the key array; cntw: of this warp's count row.
__device__ __forceinline__ bool table_count(uint32_t keys, uint32_t cntw, uint32_t K) {
  const uint32_t h = ((K ^ (K >> 15)) * 0x9e3779b1u) >> (32 - kNTBits);
  for (int p = 0; p < kProbe; ++p) {
    const uint32_t s = (h + p) & (kNT - 1);
    uint32_t cur = lds_volatile_u32(keys + 4 * s);
    if (cur == kNoKey) cur = atoms_cas_u32(keys + 4 * s, kNoKey, K);
    if (cur == kNoKey || cur == K) {
      reds_add_u32(cntw + 4 * s, 1u);
      return true;
    }
  }
  return false;
}

// Step 2: exact mass above and below classes [lo, hi]; keys inside counted.
// Returns 1 if the table overflowed.
template <int DT>
__device__ __noinline__ int topp_exact_pass(const Row row, float m, float cT, uint64_t ck, Level L, int lo,
                                            int hi, Smem& sm, FullExtra& fx, double& above, double& below) {
  constexpr int P = Elem<DT>::kPer;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  fx.u.t.keys[tid] = kNoKey;
#pragma unroll
  for (int w = 0; w < kWarps; ++w) fx.u.t.cnt[w][tid] = 0u;
  if (tid == 0) fx.bi[0] = 0;
  __syncthreads();
  volatile int* ovf = &fx.bi[0];
  const uint32_t keys = smem_u32(fx.u.t.keys), cntw = smem_u32(fx.u.t.cnt[warp]);
  float sa = 0.0f, ca = 0.0f, sb = 0.0f, cb = 0.0f;
  const int Ls = seg_len(row);
  const int v0 = warp * Ls, v1 = min(row.nvec, v0 + Ls);
  for (int s = v0; s < v1; s += 32 * kUnroll) {
    if (*ovf) break;
    uint4 r[kUnroll];
    int c[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = s + u * 32 + lane;
      c[u] = v < v1 ? load_vec<DT, false>(row, v, r[u]) : 0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      if (c[u] == 0) continue;
      float x[P];
      unpack<DT>(r[u], x);
      const int v = s + u * 32 + lane;
#pragma unroll
      for (int e = 0; e < P; ++e) {
        if (e >= c[u]) continue;
        const uint32_t K = fkey(x[e]);
        if (ck != 0ull && composite(K, static_cast<uint32_t>(v * P + e)) < ck) continue;
        const float t = (x[e] - m) * cT;
        const int cl = class_of(t, L);
        const float w = fast_exp2(t);
        const bool up = cl < lo, down = cl > hi;
        kahan_add(sa, ca, up ? w : 0.0f);      // branch-free: both sums see every element
        kahan_add(sb, cb, down ? w : 0.0f);
        if (!up && !down && !table_count(keys, cntw, K)) *ovf = 1;
      }
    }
  }
  above = block_sum_d(static_cast<double>(sa) - static_cast<double>(ca), sm);
  below = block_sum_d(static_cast<double>(sb) - static_cast<double>(cb), sm);
  return fx.bi[0];
}

// Step 3: crossing key, ties taken and W from the table; the cut's index from
// one warp segment.  False if the bracket does not hold the crossing.
template <int DT>
__device__ __noinline__ bool topp_resolve(const Row row, float m, float cT, float top_p, double above,
                                          double below, Smem& sm, FullExtra& fx, uint64_t& cut, double& W) {
  auto& T = fx.u.t;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t K = T.keys[tid];
  const bool valid = K != kNoKey;
  double mass = 0.0;
  if (valid) {
    uint32_t count = 0;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) count += T.cnt[w][tid];
    const float wK = fast_exp2((key_value(K) - m) * cT);   // the weight every element of key K got
    mass = static_cast<double>(count) * static_cast<double>(wK);
    int rank = 0;
    for (int s = 0; s < kNT; ++s) {
      const uint32_t o = T.keys[s];
      rank += (o != kNoKey && o > K) ? 1 : 0;
    }
    T.skey[rank] = K;
    T.scnt[rank] = count;
    T.sw[rank] = wK;
    T.smass[rank] = mass;
    T.sslot[rank] = static_cast<int16_t>(tid);
  }
  const int nk = __syncthreads_count(valid);
  const double inb = block_sum_d(mass, sm);
  const double tau = static_cast<double>(top_p) * (above + below + inb);
  if (!(nk > 0 && above < tau && tau <= above + inb)) return false;   // same values in every thread
  if (warp == 0) {
    double run = above, before = 0.0;
    int pos = -1;
    for (int base = 0; base < nk; base += 32) {
      const int i = base + lane;
      const double ms = i < nk ? T.smass[i] : 0.0;
      const double incl = warp_incl_scan_f64(ms, lane);
      const unsigned bal = __ballot_sync(kFull, i < nk && run + incl >= tau);
      if (bal) {
        const int Lb = __ffs(bal) - 1;
        pos = base + Lb;
        before = run + __shfl_sync(kFull, incl - ms, Lb);
        break;
      }
      run += __shfl_sync(kFull, incl, 31);
    }
    if (pos < 0) {                          // rounding left tau just above the scanned total
      pos = nk - 1;
      before = run - T.smass[pos];
    }
    if (lane == 0) {
      const double wk = static_cast<double>(T.sw[pos]);
      double need = ceil((tau - before) / wk);
      if (!(need >= 1.0)) need = 1.0;
      if (need > static_cast<double>(T.scnt[pos])) need = static_cast<double>(T.scnt[pos]);
      const uint32_t n = static_cast<uint32_t>(need);
      fx.bd[0] = before + need * wk;
      const int slot = T.sslot[pos];
      uint32_t acc = 0, r = n;
      int Wn = kWarps - 1;
      for (int w = 0; w < kWarps; ++w) {
        const uint32_t cw = T.cnt[w][slot];
        if (acc + cw >= n) { Wn = w; r = n - acc; break; }
        acc += cw;
      }
      fx.bi[1] = static_cast<int>(T.skey[pos]);
      fx.bi[2] = Wn;
      fx.bi[3] = static_cast<int>(r);
    }
  }
  __syncthreads();
  const uint32_t Ks = static_cast<uint32_t>(fx.bi[1]);
  const int Ls = seg_len(row), v0 = min(row.nvec, fx.bi[2] * Ls);
  const int idx = range_find_nth<DT>(row, Ks, v0, min(row.nvec, v0 + Ls), static_cast<uint32_t>(fx.bi[3]), sm);
  if (idx < 0) return false;
  cut = composite(Ks, static_cast<uint32_t>(idx));
  W = fx.bd[0];
  return true;
}

// The top-p cut among {composite >= ck} by bracketing; false if it gave up.
template <int DT>
__device__ __noinline__ bool topp_bracketed(const Row row, float m, float cT, uint64_t ck, float top_p,
                                            Smem& sm, FullExtra& fx, uint64_t& cut, double& W) {
  Level L;
  L.top = 0.0f;
  float w = kLevel0Width;
  L.inv_w = 1.0f / w;
  for (int level = 0; level < kMaxLevels; ++level) {
    topp_bucket_pass<DT>(row, m, cT, ck, L, sm, fx);
    int lo, hi;
    choose_bracket(fx.csum, top_p, lo, hi);
    double above, below;
    const int overflow = topp_exact_pass<DT>(row, m, cT, ck, L, lo, hi, sm, fx, above, below);
    if (!overflow) return topp_resolve<DT>(row, m, cT, top_p, above, below, sm, fx, cut, W);
    if (lo == 0) return false;              // nothing above the range to refine into
    L.top = L.top - static_cast<float>(lo - 1) * w;
    if (hi <= kNB) w = w * static_cast<float>(hi - lo + 1) / static_cast<float>(kNB);
    L.inv_w = 1.0f / w;
  }
  return false;
}

// 16-bit order key of bf16 bits b (-0 folded onto +0), and back.
__device__ __forceinline__ uint32_t bf16_key(uint32_t b) {
  b = (b == 0x8000u) ? 0u : b;
  return (b & 0x8000u) ? (~b & 0xffffu) : (b | 0x8000u);
}
__device__ __forceinline__ float bf16_key_value(uint32_t k) {
  const uint32_t b = (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu);
  return __uint_as_float(b << 16);
}
// bf16 bits of key-count slot s (direct window or small table).
__device__ __forceinline__ uint32_t kc_slot_bits(const KeyCount& T, int s) {
  if (s < kKCDirect) {
    const uint32_t sign = static_cast<uint32_t>(s) >> 10, rel = (static_cast<uint32_t>(s) >> 7) & 7u;
    return (sign << 15) | ((rel + kKCExpLo) << 7) | (static_cast<uint32_t>(s) & 127u);
  }
  const uint32_t k = T.keys[s - kKCDirect];
  return (k & 0x8000u) ? (k & 0x7fffu) : (~k & 0xffffu);
}

// Direct-window slot of bf16 bits b (only bits 0..15 are read): with
// t = (exponent - kKCExpLo) * 128 + mantissa, in the window iff t < 1024, at
// slot sign * 1024 + t.  Returns t; *off = the sign's byte offset (4 * 1024).
__device__ __forceinline__ uint32_t kc_direct(uint32_t b, uint32_t& off) {
  off = (b >> 3) & 0x1000u;
  return (b & 0x7fffu) - (static_cast<uint32_t>(kKCExpLo) << 7);
}

// Counts the elements of vector words q selected by mask in the small table
// (keys: its key array); NaN / +inf set *bad, -inf is skipped (probability
// 0).  Inline, but only reached for the rare values outside the direct
// window.  False on overflow.
__device__ __forceinline__ bool kc_count_table(uint32_t keys, uint32_t cnt, uint4 q, uint32_t mask,
                                               volatile int* bad) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  while (mask) {
    const int e = __ffs(mask) - 1;
    mask &= mask - 1;
    const uint32_t b = ((e & 1) ? (w[e >> 1] >> 16) : w[e >> 1]) & 0xffffu;
    if ((b & 0x7f80u) == 0x7f80u) {                     // inf or NaN
      if (b != 0xff80u) *bad = 1;
      continue;
    }
    const uint32_t k = bf16_key(b);
    const uint32_t h = (k * 0x9e3779b1u) >> (32 - kKHBits);
    bool done = false;
    for (int p = 0; p < kKHProbe && !done; ++p) {
      const uint32_t s = (h + p) & (kKH - 1);
      uint32_t cur = lds_volatile_u32(keys + 4 * s);
      if (cur == kNoKey) cur = atoms_cas_u32(keys + 4 * s, kNoKey, k);
      if (cur == kNoKey || cur == k) {
        reds_add_u32(cnt + 4 * (kKCDirect + s), 1u);
        done = true;
      }
    }
    if (!done) return false;
  }
  return true;
}

// The counting loop of kc_pass, for aligned or element-wise rows.
template <bool kAligned>
__device__ __forceinline__ void kc_loop(const Row row, int v0, int v1, uint32_t keys, uint32_t cnt,
                                        volatile int* ovf, volatile int* bad, const StopCheck& sc,
                                        volatile int* abandoned) {
  constexpr int P = Elem<DT_BF16>::kPer;
  const int lane = threadIdx.x & 31;
  bool counting = true;   // this thread's; an overflow anywhere discards the counts
  unsigned seen = 0u;     // the stop mark as read two iterations earlier (one load per warp)
  int it = 0;
  for (int s = v0; s < v1 && counting; s += 32 * kUnroll, ++it) {
    if (sc.p && (it & 1)) {
      if (seen > sc.thr) {                             // the sequence stopped: abandon the row
        *abandoned = 1;
        break;
      }
      seen = ld_relaxed_u32(sc.p);                     // consumed two iterations later
    }
    uint4 r[kUnroll];
    int c[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int v = s + u * 32 + lane;
      r[u] = make_uint4(0u, 0u, 0u, 0u);
      c[u] = v < v1 ? load_vec_as<DT_BF16, false, kAligned>(row, v, r[u]) : 0;
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const uint32_t w[4] = {r[u].x, r[u].y, r[u].z, r[u].w};
      uint32_t rest = 0;
#pragma unroll
      for (int e = 0; e < P; ++e) {
        const uint32_t b = (e & 1) ? (w[e >> 1] >> 16) : w[e >> 1];
        uint32_t off;
        const uint32_t t = kc_direct(b, off);
        const bool valid = e < c[u], in = t < 1024u;
        reds_add_u32_if(cnt + off + 4 * t, 1u, valid && in);
        rest |= (valid && !in) ? (1u << e) : 0u;
      }
      if (__builtin_expect(rest != 0u, 0) && !kc_count_table(keys, cnt, r[u], rest, bad)) {
        *ovf = 1;
        counting = false;
      }
    }
  }
}

// Pass 1 of a bf16 top-p row: the value counts, table j for the warps of
// half j of the row; then the maximum (the largest value counted) and the
// NaN / +inf flag.  Returns 1 if the small table overflowed -- the maximum is
// then incomplete and the caller takes it with full_max.
__device__ __noinline__ int kc_pass(const Row row, Smem& sm, FullExtra& fx, float& m_out, int& bad_out,
                                    const StopCheck sc, int& abandoned) {
  const int tid = threadIdx.x, warp = tid >> 5;
  for (int s = tid; s < kKH; s += kThreads) fx.u.kc.keys[s] = kNoKey;
  for (int s = tid; s < kCountTables * kKCSlots; s += kThreads) (&fx.u.kc.cnt[0][0])[s] = 0u;
  if (tid == 0) {
    fx.bi[0] = 0;
    fx.bi[1] = 0;
    fx.bi[4] = 0;
  }
  __syncthreads();
  const uint32_t keys = smem_u32(fx.u.kc.keys), cnt = smem_u32(fx.u.kc.cnt[warp / kWarpsPerTable]);
  const int Ls = seg_len(row);
  const int v0 = warp * Ls, v1 = min(row.nvec, v0 + Ls);
  if (row.aligned) kc_loop<true>(row, v0, v1, keys, cnt, &fx.bi[0], &fx.bi[1], sc, &fx.bi[4]);
  else kc_loop<false>(row, v0, v1, keys, cnt, &fx.bi[0], &fx.bi[1], sc, &fx.bi[4]);
  __syncthreads();
  abandoned = fx.bi[4];
  if (abandoned) return 1;                             // same in every thread
  // the maximum is the largest value with a count
  const KeyCount& T = fx.u.kc;
  float m = -__int_as_float(0x7f800000);
  for (int s = tid; s < kKCSlots; s += kThreads) {
    const bool used = s < kKCDirect ? (T.cnt[0][s] | T.cnt[1][s]) != 0u : T.keys[s - kKCDirect] != kNoKey;
    if (used) m = fmaxf(m, __uint_as_float(kc_slot_bits(T, s) << 16));
  }
  static_assert(kCountTables == 2, "the used-slot test reads two count rows");
  m_out = block_max_f(m, sm);
  bad_out = fx.bi[1];
  return fx.bi[0];
}

// The cut from the value counts; false when the crossing bin holds more
// values than the list (the caller then brackets).
__device__ __noinline__ bool kc_resolve(const Row row, float m, float cT, float scale, float top_p, Smem& sm,
                                        FullExtra& fx, bool lazy, uint64_t& cut, double& W, int& ties) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const KeyCount& T = fx.u.kc;
  auto count_of = [&](int s) {
    uint32_t c = 0;
#pragma unroll
    for (int j = 0; j < kCountTables; ++j) c += T.cnt[j][s];
    return c;
  };
  auto used = [&](int s) { return s < kKCDirect ? count_of(s) != 0u : T.keys[s - kKCDirect] != kNoKey; };
  if (tid < 256) {
    sm.u.f.mass[tid] = 0ull;
    sm.u.f.cnt[tid] = 0u;
  }
  if (tid == 0) sm.ncand = 0;
  __syncthreads();
  for (int s = tid; s < kKCSlots; s += kThreads) {
    if (!used(s)) continue;
    const float t = (__uint_as_float(kc_slot_bits(T, s) << 16) - m) * cT;
    const unsigned long long wf = fixed_mass(fast_exp2(t), scale);
    const int b = tbin_of(t);
    atomicAdd(&sm.u.f.mass[b], static_cast<unsigned long long>(count_of(s)) * wf);
    atomicAdd(&sm.u.f.cnt[b], 1u);
  }
  __syncthreads();
  if (warp == 0) {
    uint64_t tot = 0;
    for (int j = lane; j < 256; j += 32) tot += sm.u.f.mass[j];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) tot += shfl_xor_u64(tot, o);
    const double tf = ceil(static_cast<double>(top_p) * static_cast<double>(tot));
    uint64_t tau = tf >= static_cast<double>(tot) ? tot : static_cast<uint64_t>(tf);
    if (tau == 0) tau = 1;
    int digit;
    uint64_t before;
    pick_digit_mass(sm.u.f.mass, 0ull, tau, false, lane, digit, before);
    if (lane == 0) {
      sm.b_u64[0] = tau;
      sm.b_u64[1] = before;
      sm.b_i32[0] = digit;
    }
  }
  __syncthreads();
  const uint64_t tau = sm.b_u64[0], above = sm.b_u64[1];
  const int tb = sm.b_i32[0];
  if (sm.u.f.cnt[tb] > static_cast<uint32_t>(kKCList)) return false;   // same in every thread
  // the crossing bin's values, as (key << 48 | slot << 32 | count), then sorted descending
  for (int s = tid; s < kKCSlots; s += kThreads) {
    if (!used(s)) continue;
    const uint32_t b = kc_slot_bits(T, s);
    if (tbin_of((__uint_as_float(b << 16) - m) * cT) != tb) continue;
    const int pos = atomicAdd(&sm.ncand, 1);
    sm.cand[pos] = (static_cast<uint64_t>(bf16_key(b)) << 48) | (static_cast<uint64_t>(s) << 32) | count_of(s);
  }
  __syncthreads();
  const int n = sm.ncand;
  for (int e = tid; e < n; e += kThreads) {
    const uint64_t c = sm.cand[e];
    int rank = 0;
    for (int j = 0; j < n; ++j) rank += sm.cand[j] > c ? 1 : 0;
    sm.cand[kKCList + rank] = c;
  }
  __syncthreads();
  if (warp == 0) {
    const uint64_t* srt = sm.cand + kKCList;
    uint64_t run = above, before = 0;
    int pos = -1;
    auto mass_of = [&](uint64_t e, unsigned long long& wf) {
      wf = fixed_mass(fast_exp2((bf16_key_value(static_cast<uint32_t>(e >> 48)) - m) * cT), scale);
      return static_cast<uint64_t>(static_cast<uint32_t>(e)) * wf;
    };
    for (int base = 0; base < n; base += 32) {
      const int i = base + lane;
      unsigned long long wf;
      const uint64_t ms = i < n ? mass_of(srt[i], wf) : 0ull;
      uint64_t incl = ms;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint64_t t = shfl_u64(incl, (lane - o) & 31);
        if (lane >= o) incl += t;
      }
      const unsigned bal = __ballot_sync(kFull, i < n && ms != 0 && run + incl >= tau);
      if (bal) {
        const int Lb = __ffs(bal) - 1;
        pos = base + Lb;
        before = run + shfl_u64(incl - ms, Lb);
        break;
      }
      run += shfl_u64(incl, 31);
    }
    if (pos < 0) {                                  // rounding: take the last value with mass
      pos = n - 1;
      unsigned long long wf;
      while (pos > 0 && mass_of(srt[pos], wf) == 0) --pos;
      before = run - mass_of(srt[pos], wf);
    }
    if (lane == 0) {
      const uint64_t e = srt[pos];
      unsigned long long wf;
      mass_of(e, wf);
      const uint32_t c = static_cast<uint32_t>(e);
      uint64_t need = (wf && tau > before) ? (tau - before + wf - 1) / wf : 1;
      if (need < 1) need = 1;
      if (need > c) need = c;
      const int slot = static_cast<int>((e >> 32) & 0xffffu);
      uint32_t acc = 0, r = static_cast<uint32_t>(need);
      int Q = kCountTables - 1;
      for (int j = 0; j < kCountTables; ++j) {
        const uint32_t cj = T.cnt[j][slot];
        if (acc + cj >= need) { Q = j; r = static_cast<uint32_t>(need) - acc; break; }
        acc += cj;
      }
      sm.b_u64[2] = before + need * wf;
      sm.b_i32[1] = static_cast<int>(fkey(bf16_key_value(static_cast<uint32_t>(e >> 48))));
      sm.b_i32[2] = Q;
      sm.b_i32[3] = static_cast<int>(r);
      sm.b_i32[8] = static_cast<int>(need);
      sm.b_i32[9] = static_cast<int>(c);
    }
  }
  __syncthreads();
  const uint32_t K32 = static_cast<uint32_t>(sm.b_i32[1]);
  const unsigned long long Wf = sm.b_u64[2];
  const int Ls = seg_len(row), Q = sm.b_i32[2];
  const uint32_t r = static_cast<uint32_t>(sm.b_i32[3]);
  const int need = sm.b_i32[8], nK = sm.b_i32[9];
  __syncthreads();
  W = static_cast<double>(Wf) / static_cast<double>(scale);
  if (lazy || need == nK) {
    // every tie of the cut value counted as kept; a lazy row keeps only the
    // first `need` of them in index order and leaves finding them to the draw
    cut = composite(K32, 0xffffffffu);
    ties = need == nK ? 0 : need;
    return true;
  }
  ties = 0;
  const int v0 = min(row.nvec, kWarpsPerTable * Q * Ls), v1 = min(row.nvec, v0 + kWarpsPerTable * Ls);
  const int idx = range_find_nth<DT_BF16>(row, K32, v0, v1, r, sm);
  if (idx < 0) return false;
  cut = composite(K32, static_cast<uint32_t>(idx));
  return true;
}

template <int DT>
__device__ void full_row(const Row row, const RowParams& P, int dtok, Smem& sm, const StopCheck sc = StopCheck()) {
  const int tid = threadIdx.x;
  float m;
  double S = 0.0;
  int bad;
  // top-p needs the launch's extra shared memory for key counts or bracketing
  const unsigned dyn = dyn_smem_bytes();
  const bool extra = dyn >= sizeof(Smem) + sizeof(FullExtra);            // bracketing
  FullExtra& fx = *reinterpret_cast<FullExtra*>(reinterpret_cast<unsigned char*>(&sm) + sizeof(Smem));
  const bool keycount = DT == DT_BF16 && dyn >= sizeof(Smem) + kKCExtraBytes && P.k == 0 && P.top_p < 1.0f;
  int kc_overflow = 1;
  if (keycount) {
    int abandoned = 0;
    kc_overflow = kc_pass(row, sm, fx, m, bad, sc, abandoned);
    if (abandoned) {
      abandon_row(sm, P.cT);
      return;
    }
    if (kc_overflow) full_max<DT>(row, sm, m, bad);
  }
  // the softmax denominator of the whole row is W only with neither cut
  else if (P.k > 0 || P.top_p < 1.0f) full_max<DT>(row, sm, m, bad);
  else full_pass1<DT>(row, P.cT, sm, m, S, bad);
  if (stop_now(sc, sm)) {                              // stopped during the first pass
    abandon_row(sm, P.cT);
    return;
  }
  RowStat st;
  st.path = PATH_FULL;
  st.m = m;
  st.cut = 0;
  st.n_list = 0;
  st.argmax = -1;
  st.W = S;
  st.p_tok = 0.0f;
  st.cT = P.cT;
  st.status = bad ? SEQ_NONFINITE : (m > -__int_as_float(0x7f800000) ? SEQ_OK : SEQ_EMPTY_SUPPORT);
  if (st.status == SEQ_OK) {
    const float scale = __int_as_float((127 + P.fixed_shift) << 23);   // 2^fixed_shift
    uint64_t ck = 0;
    if (P.k > 0) ck = full_select_topk<DT>(row, m, P.cT, P.k, sm);
    if (P.top_p < 1.0f) {
      // key counts, else bracketing, else the radix rounds (which need no extra memory)
      bool done = false;
      if (keycount && !kc_overflow)
        done = kc_resolve(row, m, P.cT, scale, P.top_p, sm, fx, P.lazy != 0, st.cut, st.W, st.n_list);
      if (!done && extra) done = topp_bracketed<DT>(row, m, P.cT, ck, P.top_p, sm, fx, st.cut, st.W);
      if (!done) {
        unsigned long long Wf = 0;
        st.cut = full_select_topp<DT>(row, m, P.cT, scale, ck, P.top_p, sm, Wf);
        st.W = static_cast<double>(Wf) / static_cast<double>(scale);
      }
    } else if (ck) {
      st.cut = ck;
      st.W = full_sum_kept<DT>(row, m, P.cT, ck, sm);
    }
  }
  // a lazy cut: the draft token, if it equals the cut value, is kept iff fewer
  // than n_list ties come before it (same decision in every thread)
  bool tie_kept = true;
  if (st.status == SEQ_OK && dtok >= 0 && st.n_list > 0) {
    const uint32_t K = static_cast<uint32_t>(st.cut >> 32);
    if (fkey(load_elem<DT>(row.base, dtok)) == K)
      tie_kept = count_key_before<DT>(row, K, dtok, sm) < static_cast<uint32_t>(st.n_list);
  }
  if (tid == 0) {                    // one thread forms the float64 quotients
    st.invW = st.status == SEQ_OK ? static_cast<float>(1.0 / st.W) : 0.0f;
    if (st.status == SEQ_OK && dtok >= 0) {
      const float z = load_elem<DT>(row.base, dtok);
      if (tie_kept && composite(fkey(z), static_cast<uint32_t>(dtok)) >= st.cut)
        st.p_tok = static_cast<float>(static_cast<double>(fast_exp2((z - m) * P.cT)) / st.W);
    }
    sm.st = st;
  }
  __syncthreads();
}

// ------------------------------------------------------------------ PATH_STREAM
// k-th largest (1-based) composite of the contiguous shared buffer buf[0..n),
// n > k, by a block-wide MSB-first radix select (counts in sm.u.f.cnt).
__device__ __noinline__ uint64_t block_select_kth(const uint64_t* buf, int n, int k, Smem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint64_t prefix = 0, mask = 0;
  uint32_t need = static_cast<uint32_t>(k);
  for (int shift = 56; shift >= 0; shift -= 8) {
    if (tid < 256) { sm.u.f.cnt[tid] = 0u; sm.u.f.mx[tid] = 0ull; }
    __syncthreads();
    for (int e = tid; e < n; e += kThreads) {
      const uint64_t c = buf[e];
      if ((c & mask) == prefix) {
        const int d = static_cast<int>((c >> shift) & 255u);
        atomicAdd(&sm.u.f.cnt[d], 1u);
        atomicMax(&sm.u.f.mx[d], static_cast<unsigned long long>(c));
      }
    }
    __syncthreads();
    if (warp == 0) {
      int digit;
      uint32_t before;
      pick_digit_count(sm.u.f.cnt, need, true, lane, digit, before);
      if (lane == 0) {
        sm.b_i32[0] = digit;
        sm.b_i32[1] = static_cast<int>(before);
        sm.b_i32[2] = static_cast<int>(sm.u.f.cnt[digit]);
        sm.b_u64[0] = sm.u.f.mx[digit];
      }
    }
    __syncthreads();
    const int digit = sm.b_i32[0];
    need -= static_cast<uint32_t>(sm.b_i32[1]);
    const int cd = sm.b_i32[2];
    const uint64_t mx = sm.b_u64[0];
    prefix |= static_cast<uint64_t>(digit) << shift;
    mask |= 0xffull << shift;
    __syncthreads();
    if (cd == 1) return mx;
  }
  return prefix;
}

// Appends every element of the row whose composite is >= lo into sm.cand
// (a re-read of the whole row; used only when the candidate buffer overflowed).
template <int DT>
__device__ __noinline__ void collect_at_least(const Row row, uint64_t lo, Smem& sm) {
  constexpr int P = Elem<DT>::kPer;
  if (threadIdx.x == 0) sm.ncand = 0;
  __syncthreads();
  for (int v = threadIdx.x; v < row.nvec; v += kThreads) {
    uint4 r;
    const int c = load_vec<DT, false>(row, v, r);
    float x[P];
    unpack<DT>(r, x);
#pragma unroll
    for (int e = 0; e < P; ++e) {
      if (e >= c) continue;
      const uint64_t cc = composite(fkey(x[e]), static_cast<uint32_t>(v * P + e));
      if (cc >= lo) {
        const int pos = atomicAdd(&sm.ncand, 1);
        if (pos < kCandCap) sm.cand[pos] = cc;
      }
    }
  }
  __syncthreads();
}

// From the candidates in sm.cand (a superset of the row's top-k): the exact
// top-k in descending order, then float64 softmax over them, the top-p cut
// and the kept list [wrblog §7.2, §7.3].
template <int DT>
__device__ __noinline__ void stream_finish(const Row row, const RowParams P, const int dtok,
                                           const int any_bad, float m_row, Smem& sm) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = P.k;
  int n_c = sm.ncand;
  if (!any_bad && n_c > kCandCap) {
    // adversarial row (e.g. long runs of equal logits): exact selection by radix rounds
    const uint64_t ck = full_select_topk<DT>(row, m_row, P.cT, k, sm);
    collect_at_least<DT>(row, ck, sm);
    n_c = min(sm.ncand, kCandCap);
  }
  int ntop = 0;
  const uint64_t* src = sm.cand;
  int nsrc = any_bad ? 0 : n_c;
  if (nsrc > kListCap) {        // narrow to exactly k before the register sort
    const uint64_t kth = block_select_kth(sm.cand, nsrc, k, sm);
    if (tid == 0) sm.b_i32[3] = 0;
    __syncthreads();
    for (int e = tid; e < nsrc; e += kThreads) {
      const uint64_t c = sm.cand[e];
      if (c >= kth) sm.topk[atomicAdd(&sm.b_i32[3], 1)] = c;
    }
    __syncthreads();
    src = sm.topk;
    nsrc = sm.b_i32[3];
  }
  ntop = min(nsrc, k);

  // rank sort (descending), one candidate per thread (nsrc <= kListCap <= kThreads)
  static_assert(kListCap <= kThreads, "one thread per candidate");
  if (tid < nsrc) {
    const uint64_t c = src[tid];
    const ulonglong2* src2 = reinterpret_cast<const ulonglong2*>(src);   // two composites per load
    int rank = 0;
#pragma unroll 2
    for (int j = 0; j < (nsrc >> 1); ++j) {
      const ulonglong2 e = src2[j];
      rank += (e.x > c ? 1 : 0) + (e.y > c ? 1 : 0);
    }
    if (nsrc & 1) rank += src[nsrc - 1] > c ? 1 : 0;
    if (rank < k) sm.sorted[rank] = c;
  }
  __syncthreads();

  // ---- softmax over the top-k, top-p cut, kept list (warp 0; lane takes
  // positions 4*lane .. 4*lane+3).  Each weight exp((z - m) / T) = 2^((z - m) cT)
  // is evaluated from the exact difference z - m (two-sum) and a hi/lo split of
  // the exponent, so its error is exp2f's (2 ulp); sums, prefix sums and the
  // normaliser are double-float.
  if (warp == 0) {
    uint64_t v[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] = (4 * lane + j < ntop) ? sm.sorted[4 * lane + j] : 0ull;
    const uint64_t top = ntop ? sm.sorted[0] : 0ull;
    RowStat st;
    st.path = PATH_STREAM;
    st.cut = 0;
    st.argmax = ntop ? static_cast<int>(comp_index(top)) : -1;
    const float m = ntop ? comp_value(top) : -__int_as_float(0x7f800000);
    st.m = m;
    st.status = any_bad ? SEQ_NONFINITE
                        : ((ntop == 0 || !(m > -__int_as_float(0x7f800000))) ? SEQ_EMPTY_SUPPORT : SEQ_OK);
    st.W = 0.0;                                               // PATH_FULL rows only
    st.p_tok = 0.0f;
    st.n_list = 0;
    st.cT = P.cT;
    st.invW = 0.0f;
    if (st.status == SEQ_OK) {
      float w[4];
      df s = df_from(0.0f);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        w[j] = (4 * lane + j < ntop) ? exp2_diff(comp_value(v[j]), m, P.cT, P.cT_lo) : 0.0f;
        s = df_add(s, df_from(w[j]));
      }
      const df incl = warp_incl_scan_df(s, lane);
      // W = the kept weights' sum: the cumulative sum through the last kept
      // position (all of them without a top-p cut)
      df W = df_shfl(incl, 31);
      int n_keep = ntop;
      if (P.top_p < 1.0f) {
        const df S = W;
        const float th = P.top_p * S.hi;                       // target = top_p * S, double-float
        const df target = {th, fmaf(P.top_p, S.hi, -th) + P.top_p * S.lo};
        df acc = df_shfl_up(incl, 1);                          // exclusive prefix of this lane
        if (lane == 0) acc = df_from(0.0f);
        int first = 0x7fffffff;
        df at_first = S;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int pos = 4 * lane + j;
          if (pos < ntop) {
            acc = df_add(acc, df_from(w[j]));
            if (first == 0x7fffffff && df_ge(acc, target)) {
              first = pos;
              at_first = acc;
            }
          }
        }
        const unsigned fb = __ballot_sync(kFull, first != 0x7fffffff);   // positions are lane-blocked
        if (fb) {
          const int L = __ffs(fb) - 1;
          n_keep = __shfl_sync(kFull, first, L) + 1;
          W = df_shfl(at_first, L);
        }
      }
      // 1 / W as a double-float: a float reciprocal refined by one Newton step
      // (the float64 pipe is far slower than the float pipe on this part)
      const float r = __frcp_rn(W.hi);
      const float r_lo = r * (fmaf(-W.hi, r, 1.0f) - W.lo * r);
      int hit = -1;
      float ptok = 0.0f;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int pos = 4 * lane + j;
        if (pos < n_keep) {
          const int tok = static_cast<int>(comp_index(v[j]));
          const float ph = w[j] * r;                            // p = w / W, double-float
          const float pl = fmaf(w[j], r, -ph) + w[j] * r_lo;
          const float hi = ph + pl;
          sm.list_tok[pos] = tok;
          sm.list_ph[pos] = hi;
          sm.list_pl[pos] = pl - (hi - ph);
          if (tok == dtok) { hit = lane; ptok = hi; }
        } else if (pos < ((n_keep + 3) & ~3)) {
          sm.list_tok[pos] = 0x7fffffff;                        // pad for the 4-wide rank loop
        }
      }
      const unsigned hb = __ballot_sync(kFull, hit >= 0);
      if (hb) ptok = __shfl_sync(kFull, ptok, __ffs(hb) - 1);
      st.p_tok = hb ? ptok : 0.0f;
      st.n_list = n_keep;
    }
    if (lane == 0) sm.st = st;
  }
  __syncthreads();
}

// Appends the elements of vector v whose key is >= K to sm.cand (c = valid count).
template <int DT>
__device__ __forceinline__ void append_from_vector(const uint4& r, int c, int v, uint32_t K, Smem& sm) {
  constexpr int P = Elem<DT>::kPer;
  float x[P];
  unpack<DT>(r, x);
#pragma unroll
  for (int e = 0; e < P; ++e) {
    const uint32_t key = fkey(x[e]);
    if (e < c && key >= K && !(x[e] != x[e])) {
      const int pos = atomicAdd(&sm.ncand, 1);
      if (pos < kCandCap) sm.cand[pos] = composite(key, static_cast<uint32_t>(v * P + e));
    }
  }
}

// Lower bound K for the k-th largest element of a row: the k-th largest of the
// per-thread maxima mk (k distinct elements reach it), found by an MSB-first
// radix select over 8-bit digits with block-wide counts (bf16 keys: the top
// 16 bits, two rounds).  sm.khist must be zero and visible (a barrier after
// the clear).  Block-wide.
template <int DT>
__device__ __forceinline__ uint32_t select_bound(uint32_t mk0, int k, Smem& sm) {
  const int tid = threadIdx.x;
  constexpr int kRounds = DT == DT_BF16 ? 2 : 4;
  uint32_t prefix = 0u;
  uint32_t need = static_cast<uint32_t>(k);
#pragma unroll
  for (int rd = 0; rd < kRounds; ++rd) {
    const int sh = 24 - 8 * rd;
    uint32_t* hist = sm.khist[rd & 1];
    if (rd == 0 || (mk0 >> (sh + 8)) == prefix) atomicAdd(&hist[(mk0 >> sh) & 0xffu], 1u);
    __syncthreads();
    if ((tid >> 5) == 0) {
      int digit;
      uint32_t before;
      pick_digit_count(hist, need, true, tid & 31, digit, before);
      if (tid == 0) {
        sm.b_i32[4] = static_cast<int>((prefix << 8) | static_cast<uint32_t>(digit));
        sm.b_i32[5] = static_cast<int>(need - before);
      }
    }
    __syncthreads();
    prefix = static_cast<uint32_t>(sm.b_i32[4]);
    need = static_cast<uint32_t>(sm.b_i32[5]);
    if (rd + 2 < kRounds) hist[tid] = 0u;           // reused two rounds later, after a barrier
  }
  return prefix << (32 - 8 * kRounds);
}

// PATH_STREAM row (1 <= k <= kSmallK).  Pass 1 streams the row from HBM once.
// Each thread keeps the keys and positions of its four largest vector maxima
// .  The k-th largest of the per-thread maxima is a lower bound K for
// the row's k-th largest element (k distinct elements reach it), found bit by
// bit with block-wide counts.  Only vectors whose maximum reaches K can hold a
// top-k element: a thread re-reads its tracked ones in one round trip, or all
// its groups when all four tracked vectors qualify (there may be more).  The
// collected elements >= K are a small superset of the top-k.
template <int DT>
__device__ void stream_row(const Row row, const RowParams& P, int dtok, Smem& sm, const StopCheck sc = StopCheck()) {
  const int tid = threadIdx.x;
  constexpr int step = kThreads * kStreamUnroll;
  const int iters = (row.nvec + step - 1) / step;
  uint32_t mk0 = 0u, mk1 = 0u, mk2 = 0u, mk3 = 0u;      // four largest vector-max keys, descending
  int mv0 = 0, mv1 = 0, mv2 = 0, mv3 = 0;               // their vector indices
  bool bad = false;
#pragma unroll
  for (int h = 0; h < 2; ++h) sm.khist[h][tid] = 0u;   // visible after the barrier below
  // One vector's contribution: its maximum, and an insertion among the four tracked.
  const auto take = [&](const uint4& r, int c, int v) {
    bool vb;
    const uint32_t vk = fkey(vec_max<DT>(r, c, vb));
    bad |= vb;
    if (vk > mk3) {                                  // insert, keeping earlier vectors first on ties
      const bool g0 = vk > mk0, g1 = vk > mk1, g2 = vk > mk2;
      mk3 = g2 ? mk2 : vk;                 mv3 = g2 ? mv2 : v;
      mk2 = g2 ? (g1 ? mk1 : vk) : mk2;   mv2 = g2 ? (g1 ? mv1 : v) : mv2;
      mk1 = g1 ? (g0 ? mk0 : vk) : mk1;   mv1 = g1 ? (g0 ? mv0 : v) : mv1;
      mk0 = g0 ? vk : mk0;                 mv0 = g0 ? v : mv0;
    }
  };
  if (row.aligned) {
    // Aligned rows: thread t takes vectors t, t + kThreads, ... through a ring of
    // kRing shared-memory slots filled by cp.async, kRing - 1 copies in flight.
    const int nk = (row.nvec - tid + kThreads - 1) / kThreads;
    const char* src = row.base + static_cast<size_t>(tid) * 16;
    constexpr size_t kStride = static_cast<size_t>(kThreads) * 16;
#pragma unroll
    for (int s = 0; s < kRing - 1; ++s) {
      if (s < nk) cp_async16(&sm.u.ring[s][tid], src + s * kStride);
      cp_async_commit();
    }
    int slot = 0, fill = kRing - 1;
    for (int k = 0; k < nk; ++k) {
      if (k + kRing - 1 < nk) cp_async16(&sm.u.ring[fill][tid], src + (k + kRing - 1) * kStride);
      cp_async_commit();
      cp_async_wait<kRing - 1>();                    // the copy of vector k has landed
      const uint4 r = sm.u.ring[slot][tid];
      slot = slot + 1 == kRing ? 0 : slot + 1;
      fill = fill + 1 == kRing ? 0 : fill + 1;
      take(r, Elem<DT>::kPer, tid + k * kThreads);
    }
    cp_async_wait<0>();
  }
  for (int it = 0; !row.aligned && it < iters; ++it) {
    uint4 r[kStreamUnroll];
    int cnt[kStreamUnroll];
#pragma unroll
    for (int u = 0; u < kStreamUnroll; ++u) cnt[u] = load_vec<DT, true>(row, it * step + u * kThreads + tid, r[u]);
#pragma unroll
    for (int u = 0; u < kStreamUnroll; ++u)
      if (cnt[u]) take(r[u], cnt[u], it * step + u * kThreads + tid);
  }
  const int any_bad = __syncthreads_or(bad ? 1 : 0);
  if (stop_now(sc, sm)) {                              // stopped while the row streamed
    abandon_row(sm, P.cT);
    return;
  }
  const uint32_t K = select_bound<DT>(mk0, P.k, sm);
  if (tid == 0) {
    sm.ncand = 0;
    sm.nfull = 0;
  }
  __syncthreads();
  if (!any_bad && mk3 != 0u && mk3 >= K) {
    // every tracked vector qualifies and more may: the CTA re-reads all of them below
    const int pos = atomicAdd(&sm.nfull, 1);
    if (pos < kMaxFull) sm.full[pos] = tid;
  } else if (!any_bad && mk0 != 0u && mk0 >= K) {
    uint4 r0, r1, r2;
    const int c0 = load_vec<DT, false>(row, mv0, r0);
    const int c1 = (mk1 != 0u && mk1 >= K) ? load_vec<DT, false>(row, mv1, r1) : 0;
    const int c2 = (mk2 != 0u && mk2 >= K) ? load_vec<DT, false>(row, mv2, r2) : 0;
    append_from_vector<DT>(r0, c0, mv0, K, sm);
    if (c1) append_from_vector<DT>(r1, c1, mv1, K, sm);
    if (c2) append_from_vector<DT>(r2, c2, mv2, K, sm);
  }
  __syncthreads();
  const int nfull = sm.nfull;
  if (nfull > 0) {
    // cooperative re-read: one vector per job, jobs spread over the whole CTA
    const int per = (row.nvec + kThreads - 1) / kThreads;       // vectors per thread
    const bool all = nfull > kMaxFull;                           // too many: re-read the whole row
    if (all) {                       // the whole row is re-read: drop what the tracked vectors added
      if (tid == 0) sm.ncand = 0;
      __syncthreads();
    }
    const int jobs = all ? row.nvec : nfull * per;
    for (int job = tid; job < jobs; job += kThreads) {
      const int v = all ? job : sm.full[job / per] + (job % per) * kThreads;
      uint4 r;
      const int c = load_vec<DT, false>(row, v, r);
      if (c) append_from_vector<DT>(r, c, v, K, sm);
    }
    __syncthreads();
  }
  stream_finish<DT>(row, P, dtok, any_bad, 0.0f, sm);
}

// PATH_STREAM row for 16-byte aligned rows: stream_row's analysis with a
// leaner streaming loop.  Thread t takes vectors t, t + kThreads, ... through
// its cp.async ring of kRing slots and tracks its four largest vector maxima
// (order keys and positions).  At five row CTAs per SM the stream is close to
// bound by instruction issue, and the warp schedulers then favour the oldest
// warps, so every instruction per vector slows the last rows most: the ring is
// unrolled by its depth (constant slots), addresses advance by one add, the
// vector maximum's key is vec_max_okey's, and the NaN / +inf test is made
// once, on the largest key.  Nothing is written to shared memory while the
// thread's copies are in flight (a shared store or atomic then waits for
// them).  After the bound K is known each thread re-reads its qualifying
// tracked vectors in one round trip; if the fourth tracked maximum reaches K
// the thread may hold more qualifying vectors than it tracked, and the block
// re-reads all of them.  (Keeping the three best vectors in registers instead
// of re-reading them measured slower: the register moves ride on the
// insertion that nearly every warp-iteration takes.)  The draft token whose
// probability the row reports comes from dtok_of(), called by every thread
// once the stream is done (the caller may wait for a previous grid there).
template <int DT, class DtokOf>
__device__ void lean_stream_row(const Row row, const RowParams& P, DtokOf dtok_of, Smem& sm) {
  static_assert(kRing == 4, "the loop below is unrolled for four slots");
  constexpr uint32_t kSlot = kThreads * 16;                 // bytes per ring slot
  constexpr size_t kStride = static_cast<size_t>(kThreads) * 16;
  const int tid = threadIdx.x;
  uint32_t mk0 = 0u, mk1 = 0u, mk2 = 0u, mk3 = 0u;      // four largest vector-max keys, descending
  int mv0 = 0, mv1 = 0, mv2 = 0, mv3 = 0;               // their vector indices
#pragma unroll
  for (int h = 0; h < 2; ++h) sm.khist[h][tid] = 0u;   // visible after the barrier below
  const int nk = (row.nvec - tid + kThreads - 1) / kThreads;
  const uint32_t rs = smem_u32(&sm.u.ring[0][tid]);      // slot s of this thread: rs + s kSlot
  const char* gp = row.base + static_cast<size_t>(tid) * 16;
#pragma unroll
  for (int s = 0; s < kRing - 1; ++s) {
    if (s < nk) cp_async16_to(rs + s * kSlot, gp + s * kStride);
    cp_async_commit();
  }
  gp += (kRing - 1) * kStride;                           // the next vector to copy: k + 3
  // one vector: its maximum's key, and an insertion among the tracked four
  // (earlier vectors stay first on ties)
  const auto take = [&](const uint4& r, int v) {
    const uint32_t vk = vec_max_okey<DT>(r);
    if (vk > mk3) {
      const bool g0 = vk > mk0, g1 = vk > mk1, g2 = vk > mk2;
      mk3 = g2 ? mk2 : vk;                 mv3 = g2 ? mv2 : v;
      mk2 = g2 ? (g1 ? mk1 : vk) : mk2;   mv2 = g2 ? (g1 ? mv1 : v) : mv2;
      mk1 = g1 ? (g0 ? mk0 : vk) : mk1;   mv1 = g1 ? (g0 ? mv0 : v) : mv1;
      mk0 = g0 ? vk : mk0;                 mv0 = g0 ? v : mv0;
    }
  };
  int k = 0;
  for (; k + 2 * kRing - 1 <= nk; k += kRing) {          // every copy issued below is in range
#pragma unroll
    for (int j = 0; j < kRing; ++j) {
      cp_async16_to(rs + ((j + kRing - 1) & (kRing - 1)) * kSlot, gp);
      gp += kStride;
      cp_async_commit();
      cp_async_wait<kRing - 1>();                        // the copy of vector k + j has landed
      take(lds128(rs + j * kSlot), tid + (k + j) * kThreads);
    }
  }
  for (; k < nk; ++k) {
    if (k + kRing - 1 < nk) {
      cp_async16_to(rs + ((k + kRing - 1) & (kRing - 1)) * kSlot, gp);
      gp += kStride;
    }
    cp_async_commit();
    cp_async_wait<kRing - 1>();
    take(lds128(rs + (k & (kRing - 1)) * kSlot), tid + k * kThreads);
  }
  cp_async_wait<0>();
  // a NaN or +inf anywhere in the thread's vectors puts its largest key at or above +inf's
  const int any_bad = __syncthreads_or(mk0 >= kOkeyPosInf ? 1 : 0);
  const uint32_t K = select_bound<DT>(mk0, P.k, sm);     // order-key bound
  const uint32_t Kf = fkey_of_okey(K);                   // the same bound on fkey's scale
  if (tid == 0) {
    sm.ncand = 0;
    sm.nfull = 0;
  }
  __syncthreads();
  if (!any_bad && mk3 != 0u && mk3 >= K) {
    // every tracked vector qualifies and more may: the CTA re-reads all of them below
    const int pos = atomicAdd(&sm.nfull, 1);
    if (pos < kMaxFull) sm.full[pos] = tid;
  } else if (!any_bad && mk0 != 0u && mk0 >= K) {
    uint4 r0, r1, r2;
    const int c0 = load_vec<DT, false>(row, mv0, r0);
    const int c1 = (mk1 != 0u && mk1 >= K) ? load_vec<DT, false>(row, mv1, r1) : 0;
    const int c2 = (mk2 != 0u && mk2 >= K) ? load_vec<DT, false>(row, mv2, r2) : 0;
    append_from_vector<DT>(r0, c0, mv0, Kf, sm);
    if (c1) append_from_vector<DT>(r1, c1, mv1, Kf, sm);
    if (c2) append_from_vector<DT>(r2, c2, mv2, Kf, sm);
  }
  __syncthreads();
  const int nfull = sm.nfull;
  if (nfull > 0) {
    // cooperative re-read: one vector per job, jobs spread over the whole CTA
    const int per = (row.nvec + kThreads - 1) / kThreads;       // vectors per thread
    const bool all = nfull > kMaxFull;                           // too many: re-read the whole row
    if (all) {                       // the whole row is re-read: drop what the registers added
      if (tid == 0) sm.ncand = 0;
      __syncthreads();
    }
    const int jobs = all ? row.nvec : nfull * per;
    for (int job = tid; job < jobs; job += kThreads) {
      const int v = all ? job : sm.full[job / per] + (job % per) * kThreads;
      uint4 r;
      const int c = load_vec<DT, false>(row, v, r);
      if (c) append_from_vector<DT>(r, c, v, Kf, sm);
    }
    __syncthreads();
  }
  stream_finish<DT>(row, P, dtok_of(), any_bad, 0.0f, sm);
}

// Probability of token x under a PATH_FULL row given its logit z.
// The kept-set test composite(key(z), x) >= cut as float and index compares:
// kept iff z > v, or z == v and x <= i (cut 0 keeps everything).
struct CutTest {
  float v;
  uint32_t i;
};
__device__ __forceinline__ CutTest cut_test(uint64_t cut) {
  CutTest c;
  if (cut == 0ull) {
    c.v = -__int_as_float(0x7f800000);
    c.i = 0xffffffffu;
  } else {
    c.v = key_value(static_cast<uint32_t>(cut >> 32));
    c.i = ~static_cast<uint32_t>(cut);
  }
  return c;
}
__device__ __forceinline__ float full_prob(float z, uint32_t x, const CutTest& ct, float m, float cT, float invW) {
  const bool kept = z > ct.v || (z == ct.v && x <= ct.i);
  return kept ? fast_exp2((z - m) * cT) * invW : 0.0f;
}

}  // namespace sv
