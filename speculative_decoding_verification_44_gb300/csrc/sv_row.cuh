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
//     maximum and the softmax denominator (per-thread online rescaling,
//     Kahan-compensated float sums, float64 across threads).  A top-k or
//     top-p cut is then found by MSB-first radix selection over re-reads of
//     the row (L2-resident after pass 1): digit histograms of counts (top-k)
//     or of exact 64-bit fixed-point probability masses (top-p), the first
//     top-p round bucketed by log-probability so that hot buckets spread.
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
};

// Per-row result, mirrored into the workspace for the sequence epilogue.
struct __align__(16) RowStat {
  double W;        // normaliser: sum over the kept set of exp((z - m) / T)
  double p_tok;    // probability of the draft token this row scores (0 if none)
  uint64_t cut;    // PATH_FULL: token kept iff composite >= cut (0 keeps all)
  float m;         // row maximum
  int32_t status;  // SEQ_OK, SEQ_NONFINITE or SEQ_EMPTY_SUPPORT
  int32_t n_list;  // PATH_STREAM: kept-list length
  int32_t path;
  int32_t argmax;  // greedy rows: argmax token
  int32_t pad;
};
static_assert(sizeof(RowStat) == 48, "RowStat layout");

struct __align__(16) ListEntry {  // one kept token of a PATH_STREAM row
  double p;
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
  double w[2 * kListCap];            // candidate weights (list-based draw)
  int32_t tok[2 * kListCap];
  double sw[2 * kListCap];           // sorted by token
  int32_t stok[2 * kListCap];
  int32_t qtok[kListCap];            // draft kept list sorted by token (binary search)
  double qp[kListCap];
  double wtot[kWarps];               // per-warp segment totals of the block scan
  RowStat rs[2 * kMaxGamma + 1];     // the sequence's row summaries
  int32_t dtok[kMaxGamma];
  float uacc[kMaxGamma];
};
struct __align__(16) Smem {
  union {
    SmemFull f;
    SmemEpi e;
  } u;
  uint64_t cand[kCandCap];           // PATH_STREAM: candidates (composites >= the lower bound)
  uint64_t topk[kSmallK];
  uint64_t sorted[kSmallK];          // PATH_STREAM: top-k in descending order
  int32_t list_tok[kListCap];
  double list_p[kListCap];
  int nw[kWarps];
  int ncand;
  int nfull;                         // PATH_STREAM: threads whose vectors need a full re-read
  int16_t full[kMaxFull];
  uint32_t tmax[kThreads];           // PATH_STREAM: per-thread maxima (keys)
  float red_f[kWarps];
  double red_d[kWarps];
  uint64_t red_u[kWarps];
  int red_i[kWarps];
  int flag_bad;
  // broadcast slots
  uint64_t b_u64[4];
  double b_f64[4];
  int b_i32[8];
  RowStat st;
};

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
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_f64(v);
  if (lane == 0) sm.red_d[warp] = v;
  __syncthreads();
  double r = 0.0;
  for (int w = 0; w < kWarps; ++w) r += sm.red_d[w];
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
template <int DT>
__device__ void greedy_row(const Row& row, Smem& sm, int& argmax, int& status) {
  constexpr int P = Elem<DT>::kPer;
  const int tid = threadIdx.x;
  float best = -__int_as_float(0x7f800000);
  int best_i = -1;
  bool bad = false;
  for (int base = 0; base < row.nvec; base += kThreads * kUnroll) {
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
__device__ void full_pass1(const Row& row, float cT, Smem& sm, float& m_out, double& S_out, int& bad_out) {
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
__device__ __noinline__ double full_sum_kept(const Row& row, float m, float cT, uint64_t cut, Smem& sm) {
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
  return block_sum_d(static_cast<double>(s), sm);
}

// Index of the n-th (1-based) element, in index order, whose key equals K.
template <int DT>
__device__ __noinline__ int find_nth_with_key(const Row& row, uint32_t K, uint32_t n, Smem& sm) {
  constexpr int P = Elem<DT>::kPer;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int L = (row.nvec + kWarps - 1) / kWarps;
  const int v0 = warp * L, v1 = min(row.nvec, v0 + L);
  uint32_t my = 0;
  for (int s = v0; s < v1; s += 32) {
    const int v = s + lane;
    uint4 r;
    const int c = v < v1 ? load_vec<DT, false>(row, v, r) : 0;
    if (c) {
      float x[P];
      unpack<DT>(r, x);
#pragma unroll
      for (int e = 0; e < P; ++e) my += (e < c && fkey(x[e]) == K) ? 1u : 0u;
    }
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) my += __shfl_xor_sync(kFull, my, o);
  if (lane == 0) sm.u.f.wcnt[warp] = my;
  __syncthreads();
  if (tid == 0) {
    uint32_t acc = 0;
    int W = kWarps - 1;
    uint32_t r = n;
    for (int w = 0; w < kWarps; ++w) {
      if (acc + sm.u.f.wcnt[w] >= n) { W = w; r = n - acc; break; }
      acc += sm.u.f.wcnt[w];
    }
    sm.b_i32[4] = W;
    sm.b_i32[5] = static_cast<int>(r);
    sm.b_i32[6] = -1;
  }
  __syncthreads();
  if (warp == sm.b_i32[4]) {
    const uint32_t r = static_cast<uint32_t>(sm.b_i32[5]);
    uint32_t running = 0;
    for (int s = v0; s < v1; s += 32) {
      const int v = s + lane;
      uint4 rr;
      const int c = v < v1 ? load_vec<DT, false>(row, v, rr) : 0;
      float x[P];
      unpack<DT>(rr, x);
      uint32_t mine = 0;
#pragma unroll
      for (int e = 0; e < P; ++e) mine += (e < c && fkey(x[e]) == K) ? 1u : 0u;
      const uint32_t incl = warp_incl_scan_u32(mine, lane);
      const unsigned bal = __ballot_sync(kFull, running + incl >= r && mine > 0);
      if (bal) {
        const int Lw = __ffs(bal) - 1;
        if (lane == Lw) {
          uint32_t cur = running + incl - mine;
#pragma unroll
          for (int e = 0; e < P; ++e) {
            if (e < c && fkey(x[e]) == K) {
              ++cur;
              if (cur == r) { sm.b_i32[6] = v * P + e; break; }
            }
          }
        }
        break;
      }
      running += __shfl_sync(kFull, incl, 31);
    }
  }
  __syncthreads();
  return sm.b_i32[6];
}

// One radix round over a re-read of the row.  Elements taking part: composite
// >= ck, and (if tb >= 0) in log-probability bucket tb, and matching prefix
// under mask.  kind 0: digit = bucket of log-probability; kind 1: digit = the
// composite byte at `shift`.  Accumulates counts, fixed-point masses (when
// with_mass) and the largest composite per digit.
template <int DT>
__device__ __noinline__ void full_round(const Row& row, float m, float cT, float scale, uint64_t ck, int tb,
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
__device__ __noinline__ uint64_t full_select_topk(const Row& row, float m, float cT, int k, Smem& sm) {
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
__device__ __noinline__ uint64_t full_select_topp(const Row& row, float m, float cT, float scale, uint64_t ck,
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

template <int DT>
__device__ void full_row(const Row& row, const RowParams& P, int dtok, Smem& sm) {
  const int tid = threadIdx.x;
  float m;
  double S;
  int bad;
  full_pass1<DT>(row, P.cT, sm, m, S, bad);
  RowStat st;
  st.path = PATH_FULL;
  st.m = m;
  st.cut = 0;
  st.n_list = 0;
  st.argmax = -1;
  st.W = S;
  st.p_tok = 0.0;
  st.status = bad ? SEQ_NONFINITE : (m > -__int_as_float(0x7f800000) ? SEQ_OK : SEQ_EMPTY_SUPPORT);
  if (st.status == SEQ_OK) {
    const float scale = __int_as_float((127 + P.fixed_shift) << 23);   // 2^fixed_shift
    uint64_t ck = 0;
    if (P.k > 0) ck = full_select_topk<DT>(row, m, P.cT, P.k, sm);
    if (P.top_p < 1.0f) {
      unsigned long long Wf = 0;
      st.cut = full_select_topp<DT>(row, m, P.cT, scale, ck, P.top_p, sm, Wf);
      st.W = static_cast<double>(Wf) / static_cast<double>(scale);
    } else if (ck) {
      st.cut = ck;
      st.W = full_sum_kept<DT>(row, m, P.cT, ck, sm);
    }
    if (dtok >= 0) {
      const float z = load_elem<DT>(row.base, dtok);
      if (composite(fkey(z), static_cast<uint32_t>(dtok)) >= st.cut)
        st.p_tok = static_cast<double>(fast_exp2((z - m) * P.cT)) / st.W;
    }
  }
  if (tid == 0) sm.st = st;
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
__device__ __noinline__ void collect_at_least(const Row& row, uint64_t lo, Smem& sm) {
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
__device__ __noinline__ void stream_finish(const Row& row, const RowParams& P, const int dtok,
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

  // ---- sort, softmax over the top-k, top-p cut, kept list (warp 0).
  // Each weight exp((z - m) / T) = 2^((z - m) cT) is evaluated from the exact
  // difference z - m (two-sum) and a hi/lo split of the exponent, so its error
  // is exp2f's (2 ulp); sums, prefix sums and the normaliser are double-float.
  if (warp == 0) {
    // rank sort (descending), then each lane takes positions 4*lane .. 4*lane+3
    for (int e = lane; e < nsrc; e += 32) {
      const uint64_t c = src[e];
      int rank = 0;
      for (int j = 0; j < nsrc; ++j) rank += src[j] > c ? 1 : 0;
      if (rank < k) sm.sorted[rank] = c;
    }
    __syncwarp();
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
    st.W = 0.0;
    st.p_tok = 0.0;
    st.n_list = 0;
    if (st.status == SEQ_OK) {
      float w[4];
      df s = df_from(0.0f);
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        w[j] = (4 * lane + j < ntop) ? exp2_diff(comp_value(v[j]), m, P.cT, P.cT_lo) : 0.0f;
        s = df_add(s, df_from(w[j]));
      }
      const df incl = warp_incl_scan_df(s, lane);
      int n_keep = ntop;
      if (P.top_p < 1.0f) {
        const df S = df_shfl(incl, 31);
        const float th = P.top_p * S.hi;                       // target = top_p * S, double-float
        const df target = {th, fmaf(P.top_p, S.hi, -th) + P.top_p * S.lo};
        df acc = df_add(incl, {-s.hi, -s.lo});                 // exclusive prefix
        int first = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int pos = 4 * lane + j;
          if (pos < ntop) {
            acc = df_add(acc, df_from(w[j]));
            if (first == 0x7fffffff && df_ge(acc, target)) first = pos;
          }
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) first = min(first, __shfl_xor_sync(kFull, first, o));
        n_keep = first == 0x7fffffff ? ntop : first + 1;
      }
      df part = df_from(0.0f);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if (4 * lane + j < n_keep) part = df_add(part, df_from(w[j]));
      const double W = df_to_double(warp_sum_df(part));
      const double invW = 1.0 / W;
      int hit = -1;
      double ptok = 0.0;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int pos = 4 * lane + j;
        if (pos < n_keep) {
          const int tok = static_cast<int>(comp_index(v[j]));
          const double p = static_cast<double>(w[j]) * invW;
          sm.list_tok[pos] = tok;
          sm.list_p[pos] = p;
          if (tok == dtok) { hit = lane; ptok = p; }
        }
      }
      const unsigned hb = __ballot_sync(kFull, hit >= 0);
      if (hb) ptok = __shfl_sync(kFull, ptok, __ffs(hb) - 1);
      st.W = W;
      st.p_tok = hb ? ptok : 0.0;
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

// PATH_STREAM row (1 <= k <= kSmallK).  Pass 1 streams the row from HBM once.
// Each thread keeps the keys and positions of its four largest vector maxima
// .  The k-th largest of the per-thread maxima is a lower bound K for
// the row's k-th largest element (k distinct elements reach it), found bit by
// bit with block-wide counts.  Only vectors whose maximum reaches K can hold a
// top-k element: a thread re-reads its tracked ones in one round trip, or all
// its groups when all four tracked vectors qualify (there may be more).  The
// collected elements >= K are a small superset of the top-k.
template <int DT>
__device__ void stream_row(const Row& row, const RowParams& P, int dtok, Smem& sm) {
  const int tid = threadIdx.x;
  constexpr int step = kThreads * kStreamUnroll;
  const int iters = (row.nvec + step - 1) / step;
  uint32_t mk0 = 0u, mk1 = 0u, mk2 = 0u, mk3 = 0u;      // four largest vector-max keys, descending
  int mv0 = 0, mv1 = 0, mv2 = 0, mv3 = 0;               // their vector indices
  bool bad = false;
  for (int it = 0; it < iters; ++it) {
    uint4 r[kStreamUnroll];
    int cnt[kStreamUnroll];
#pragma unroll
    for (int u = 0; u < kStreamUnroll; ++u) cnt[u] = load_vec<DT, true>(row, it * step + u * kThreads + tid, r[u]);
#pragma unroll
    for (int u = 0; u < kStreamUnroll; ++u) {
      if (cnt[u]) {
        bool vb;
        const uint32_t vk = fkey(vec_max<DT>(r[u], cnt[u], vb));
        bad |= vb;
        if (vk > mk3) {                                  // insert, keeping earlier vectors first on ties
          const int v = it * step + u * kThreads + tid;
          const bool g0 = vk > mk0, g1 = vk > mk1, g2 = vk > mk2;
          mk3 = g2 ? mk2 : vk;                 mv3 = g2 ? mv2 : v;
          mk2 = g2 ? (g1 ? mk1 : vk) : mk2;   mv2 = g2 ? (g1 ? mv1 : v) : mv2;
          mk1 = g1 ? (g0 ? mk0 : vk) : mk1;   mv1 = g1 ? (g0 ? mv0 : v) : mv1;
          mk0 = g0 ? vk : mk0;                 mv0 = g0 ? v : mv0;
        }
      }
    }
  }
  sm.tmax[tid] = mk0;
  const int any_bad = __syncthreads_or(bad ? 1 : 0);
  if ((tid >> 5) == 0) {
    // one warp searches the k-th largest of the kThreads maxima, bit by bit
    const int lane = tid & 31;
    uint32_t v[kThreads / 32];
#pragma unroll
    for (int j = 0; j < kThreads / 32; ++j) v[j] = sm.tmax[j * 32 + lane];
    uint32_t K = 0u;
    for (int bit = 31; bit >= (DT == DT_BF16 ? 16 : 0); --bit) {
      const uint32_t c = K | (1u << bit);
      uint32_t n = 0;
#pragma unroll
      for (int j = 0; j < kThreads / 32; ++j) n += v[j] >= c ? 1u : 0u;
      if (__reduce_add_sync(kFull, n) >= static_cast<uint32_t>(P.k)) K = c;
    }
    if (lane == 0) {
      sm.b_i32[4] = static_cast<int>(K);
      sm.ncand = 0;
      sm.nfull = 0;
    }
  }
  __syncthreads();
  const uint32_t K = static_cast<uint32_t>(sm.b_i32[4]);
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

// Probability of token x under a PATH_FULL row given its logit z.
__device__ __forceinline__ float full_prob(float z, uint32_t x, const RowStat& st, float cT, float invW) {
  if (st.cut != 0ull && composite(fkey(z), x) < st.cut) return 0.0f;
  return fast_exp2((z - st.m) * cT) * invW;
}

}  // namespace sv
