// sv_common.cuh -- device helpers shared by the verify kernels (sm_103a).
//
// Ordering convention used everywhere (argmax, top-k, top-p): value
// descending, token index ascending.  It is realised by the 64-bit
// "composite" (monotone float key << 32) | ~index, so that a larger composite
// always means "earlier in that order" and every composite of a row is unique.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <stdint.h>

namespace sv {

constexpr int kThreads = 256;               // threads per row CTA
constexpr int kWarps = kThreads / 32;
constexpr unsigned kFull = 0xffffffffu;
constexpr int kSmallK = 128;                // streaming top-k path handles 1 <= k <= kSmallK
constexpr int kCandCap = 1024;              // streaming top-k path: candidate buffer (entries)
constexpr int kMaxFull = 32;                // streaming top-k path: threads re-read cooperatively
constexpr int kStreamUnroll = 4;            // streaming top-k path: 16-byte loads in flight per thread
constexpr int kRing = 4;                    // streaming top-k path, aligned rows: cp.async ring slots per thread
constexpr int kListCap = kSmallK;           // kept-list entries stored per row
constexpr int kMaxGamma = 63;               // largest gamma_max the sampling verifier accepts
constexpr int kUnroll = 4;                  // 16-byte loads in flight per thread
constexpr int kScanUnroll = 2;              // inverse-CDF scan: 16-byte loads in flight per lane
constexpr int kScanChunks = 64;             // inverse-CDF scan: chunk sums kept per warp

enum { DT_BF16 = 0, DT_F32 = 1 };
enum { PATH_STREAM = 0, PATH_FULL = 1 };

enum {
  SEQ_OK = 0, SEQ_BAD_LENGTH = 1, SEQ_BAD_TOKEN = 2, SEQ_BAD_UNIFORM = 3,
  SEQ_NONFINITE = 4, SEQ_EMPTY_SUPPORT = 5, SEQ_BAD_PARAMS = 6, SEQ_BAD_TREE = 7, SEQ_STALLED = 8,
  SEQ_FLAG_ZERO_Q = 0x100, SEQ_FLAG_Z_ZERO = 0x200, SEQ_FLAG_EOS = 0x400
};

template <int DT> struct Elem;
template <> struct Elem<DT_BF16> { static constexpr int kBytes = 2; static constexpr int kPer = 8; };
template <> struct Elem<DT_F32>  { static constexpr int kBytes = 4; static constexpr int kPer = 4; };

// ---------------------------------------------------------------- keys
// Monotone unsigned key of a float: x < y  <=>  key(x) < key(y) for non-NaN
// x, y; -0.0 is folded onto +0.0 first so the two compare equal.
__device__ __forceinline__ uint32_t fkey(float x) {
  uint32_t b = __float_as_uint(x);
  if (b == 0x80000000u) b = 0u;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ float key_value(uint32_t k) {
  const uint32_t b = (k & 0x80000000u) ? (k & 0x7fffffffu) : ~k;
  return __uint_as_float(b);
}
__device__ __forceinline__ uint64_t composite(uint32_t key, uint32_t idx) {
  return (static_cast<uint64_t>(key) << 32) | static_cast<uint32_t>(~idx);
}
__device__ __forceinline__ uint32_t comp_index(uint64_t c) { return ~static_cast<uint32_t>(c); }
__device__ __forceinline__ float comp_value(uint64_t c) { return key_value(static_cast<uint32_t>(c >> 32)); }

__device__ __forceinline__ bool finite_ok(float x) { return x < __int_as_float(0x7f800000); }  // false for NaN, +inf

// 2^t with the SFU (relative error about 2^-22); 0 for t = -inf.
__device__ __forceinline__ float fast_exp2(float t) {
  float r;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(t));
  return r;
}

// exp((z - m) / T) written as 2^((z - m) cT) with cT = cT_hi + cT_lo.  The
// difference d = z - m is carried exactly as d_hi + d_lo (two-sum) and the
// exponent as t_hi + t_lo, so the only significant error left is exp2f's own
// (2 ulp): 2^(t_hi + t_lo) = 2^t_hi (1 + t_lo ln 2) to first order in t_lo.
__device__ __forceinline__ float exp2_diff(float z, float m, float cT_hi, float cT_lo) {
  const float d = z - m;                      // two-sum of z + (-m): d + d_lo == z - m exactly
  const float bb = d - z;
  const float d_lo = (z - (d - bb)) + (-m - bb);
  const float t = d * cT_hi;
  const float t_lo = fmaf(d, cT_hi, -t) + fmaf(d, cT_lo, d_lo * cT_hi);
  const float e = exp2f(t);
  return fmaf(e, t_lo * 0.6931471805599453f, e);
}

// ---------------------------------------------------------------- shared memory by address
// Explicit shared-window accesses for code that only holds a generic pointer
// (out-of-line functions): no generic-to-shared resolution per access, and
// red.shared returns nothing, so the issuing thread does not wait on it.
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ float lds_f32(uint32_t a) {
  float v;
  asm volatile("ld.shared.f32 %0, [%1];" : "=f"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ void sts_f32(uint32_t a, float v) {
  asm volatile("st.shared.f32 [%0], %1;" ::"r"(a), "f"(v) : "memory");
}
__device__ __forceinline__ uint32_t lds_volatile_u32(uint32_t a) {
  uint32_t v;
  asm volatile("ld.volatile.shared.u32 %0, [%1];" : "=r"(v) : "r"(a) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t atoms_cas_u32(uint32_t a, uint32_t cmp, uint32_t val) {
  uint32_t old;
  asm volatile("atom.shared.cas.b32 %0, [%1], %2, %3;" : "=r"(old) : "r"(a), "r"(cmp), "r"(val) : "memory");
  return old;
}
__device__ __forceinline__ void reds_add_u32(uint32_t a, uint32_t v) {
  asm volatile("red.shared.add.u32 [%0], %1;" ::"r"(a), "r"(v) : "memory");
}
// red.shared only where pred holds: a predicated instruction, no branch.
__device__ __forceinline__ void reds_add_u32_if(uint32_t a, uint32_t v, bool pred) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %2, 0;\n\t@p red.shared.add.u32 [%0], %1;\n\t}"
      ::"r"(a), "r"(v), "r"(static_cast<uint32_t>(pred)) : "memory");
}

// ---------------------------------------------------------------- loads
// Streaming 16-byte load: read once, do not keep in L1, ask L2 to fetch 256 B.
__device__ __forceinline__ uint4 ld_stream(const void* p) {
  uint4 r;
  asm("ld.global.nc.L1::no_allocate.L2::256B.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}
// Asynchronous 16-byte global -> shared copy (L1 bypassed, L2 fetches 256 B).
__device__ __forceinline__ void cp_async16(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;" :: "r"(s), "l"(gmem) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" :: "n"(N) : "memory"); }
// Asynchronous 4-byte global -> shared copy (both addresses 4-byte aligned).
__device__ __forceinline__ void cp_async4(void* smem, const void* gmem) {
  const unsigned s = static_cast<unsigned>(__cvta_generic_to_shared(smem));
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" :: "r"(s), "l"(gmem) : "memory");
}

// Arrival on a counter in global memory with release-acquire semantics at GPU
// scope (one thread of the CTA, after a barrier): writes the CTA made before
// the barrier are visible to whoever later reads the count, and the thread
// that reads the final count sees every earlier arriver's writes.
__device__ __forceinline__ unsigned atom_add_acq_rel_gpu(unsigned* p, unsigned v) {
  unsigned old;
  asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Re-read load (second pass over a row that should still sit in L2).
__device__ __forceinline__ uint4 ld_reread(const void* p) {
  uint4 r;
  asm("ld.global.nc.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w) : "l"(p));
  return r;
}

// A row is processed as "virtual vectors" of Elem<DT>::kPer consecutive
// elements.  In aligned mode (row start 16-byte aligned and vocab a multiple
// of kPer) every vector is one 16-byte load; otherwise the elements are
// fetched one by one and the last vector may be partial.
struct Row {
  const char* base;
  int V;
  int nvec;
  bool aligned;
};

template <int DT>
__device__ __forceinline__ Row make_row(const void* base, int V, bool aligned) {
  Row r;
  r.base = static_cast<const char*>(base);
  r.V = V;
  r.nvec = (V + Elem<DT>::kPer - 1) / Elem<DT>::kPer;
  r.aligned = aligned;
  return r;
}

// Loads virtual vector v; returns the number of valid elements (0 if v is past the end).
template <int DT, bool kStream>
__device__ __forceinline__ int load_vec(const Row row, int v, uint4& out) {
  constexpr int P = Elem<DT>::kPer;
  out = make_uint4(0u, 0u, 0u, 0u);
  if (v >= row.nvec) return 0;
  const int i0 = v * P;
  if (row.aligned) {
    const void* p = row.base + static_cast<size_t>(i0) * Elem<DT>::kBytes;
    out = kStream ? ld_stream(p) : ld_reread(p);
    return P;
  }
  const int n = min(P, row.V - i0);
  if (DT == DT_BF16) {
    const uint16_t* e = reinterpret_cast<const uint16_t*>(row.base) + i0;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    for (int j = 0; j < n; ++j) w[j >> 1] |= static_cast<uint32_t>(__ldg(e + j)) << ((j & 1) * 16);
    out = make_uint4(w[0], w[1], w[2], w[3]);
  } else {
    const uint32_t* e = reinterpret_cast<const uint32_t*>(row.base) + i0;
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    for (int j = 0; j < n; ++j) w[j] = __ldg(e + j);
    out = make_uint4(w[0], w[1], w[2], w[3]);
  }
  return n;
}

// load_vec for a caller that has already branched on row.aligned and
// guarantees v < row.nvec: the aligned case is one load and no branches.
template <int DT, bool kStream, bool kAligned>
__device__ __forceinline__ int load_vec_as(const Row row, int v, uint4& out) {
  if (kAligned) {
    const void* p = row.base + static_cast<size_t>(v) * 16;
    out = kStream ? ld_stream(p) : ld_reread(p);
    return Elem<DT>::kPer;
  }
  return load_vec<DT, kStream>(row, v, out);
}

// One element by index (scalar load).
template <int DT>
__device__ __forceinline__ float load_elem(const void* base, int x) {
  if (DT == DT_BF16) {
    const uint16_t b = __ldg(static_cast<const uint16_t*>(base) + x);
    return __uint_as_float(static_cast<uint32_t>(b) << 16);
  }
  return __ldg(static_cast<const float*>(base) + x);
}

template <int DT>
__device__ __forceinline__ void unpack(const uint4& r, float (&x)[Elem<DT>::kPer]) {
  if (DT == DT_BF16) {
    const uint32_t w[4] = {r.x, r.y, r.z, r.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      x[2 * j] = __uint_as_float(w[j] << 16);
      x[2 * j + 1] = __uint_as_float(w[j] & 0xffff0000u);
    }
  } else {
    x[0] = __uint_as_float(r.x);
    x[1] = __uint_as_float(r.y);
    x[2] = __uint_as_float(r.z);
    x[3] = __uint_as_float(r.w);
  }
}

// Largest value of a full vector and whether it holds a NaN or +inf.  bf16
// uses packed NaN-propagating max (three HMNMX2 for eight elements).
template <int DT>
__device__ __forceinline__ float vec_max(const uint4& r, int n, bool& bad) {
  constexpr int P = Elem<DT>::kPer;
  if (DT == DT_BF16 && n == P) {
    __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
    __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
    __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&r.z);
    __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&r.w);
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    const float lo = __low2float(m), hi = __high2float(m);
    bad = !finite_ok(lo) || !finite_ok(hi);
    return fmaxf(lo, hi);
  }
  float x[P];
  unpack<DT>(r, x);
  float m = -__int_as_float(0x7f800000);
  bool b = false;
#pragma unroll
  for (int j = 0; j < P; ++j) {
    if (j < n) {
      b |= !finite_ok(x[j]);
      m = fmaxf(m, x[j]);
    }
  }
  bad = b;
  return m;
}

// ---------------------------------------------------------------- vector maxima for the stream
// Offset-binary order key of a float's bit pattern: 2^31 plus the value's
// sign-magnitude as a signed integer, so -0 and +0 share the key 2^31.  It is
// monotone in the value, +inf maps to kOkeyPosInf and every positive-sign NaN
// above it; a bf16 value in the high half of a word keeps the key's low 16
// bits zero.  Cheaper than fkey in the streaming loop (no -0 test).
__device__ __forceinline__ uint32_t okey_bits(uint32_t bits) {
  const uint32_t s = static_cast<uint32_t>(static_cast<int32_t>(bits) >> 31);   // 0 or all ones
  return 0x80000000u + (((bits & 0x7fffffffu) ^ s) - s);
}
constexpr uint32_t kOkeyPosInf = 0xff800000u;
// The fkey of the value whose order key is k (okey_bits inverted).
__device__ __forceinline__ uint32_t fkey_of_okey(uint32_t k) {
  const uint32_t bits = k >= 0x80000000u ? (k - 0x80000000u) : (0x80000000u | (0x80000000u - k));
  return fkey(__uint_as_float(bits));
}
// Order key of the largest element of a full vector.  NaN-propagating maxima
// (max.NaN returns the canonical, positive NaN), so a vector holding a NaN or
// +inf has a key >= kOkeyPosInf.  bf16: three packed maxima, then the two
// halves against each other.
template <int DT>
__device__ __forceinline__ uint32_t vec_max_okey(const uint4& r) {
  if (DT == DT_BF16) {
    const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&r.x);
    const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&r.y);
    const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&r.z);
    const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&r.w);
    const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
    const __nv_bfloat162 mm = __hmax2_nan(m, __lowhigh2highlow(m));
    return okey_bits(*reinterpret_cast<const uint32_t*>(&mm) & 0xffff0000u);
  }
  float m;
  asm("{\n\t.reg .f32 t0, t1;\n\tmax.NaN.f32 t0, %1, %2;\n\tmax.NaN.f32 t1, %3, %4;\n\tmax.NaN.f32 %0, t0, t1;\n\t}"
      : "=f"(m) : "f"(__uint_as_float(r.x)), "f"(__uint_as_float(r.y)), "f"(__uint_as_float(r.z)),
        "f"(__uint_as_float(r.w)));
  return okey_bits(__float_as_uint(m));
}
// Programmatic dependent launch: wait until the grids this launch depends on
// have completed and their memory is visible (returns at once without such a
// dependency); allow the grids that depend on this one to be scheduled.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---------------------------------------------------------------- bulk copies
// One-dimensional global -> shared bulk copies (the copy engine, no tensor
// map) that complete on an mbarrier: one thread arms the barrier with the
// bytes to expect and issues the copies; every consumer waits on the phase.
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_init_fence() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
// bytes: a multiple of 16; both addresses 16-byte aligned.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar) : "memory");
}
// Orders this thread's earlier generic accesses to shared memory before later
// bulk copies into it (reuse of a buffer that threads have read).
__device__ __forceinline__ void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ unsigned long long global_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
// Waits for the barrier phase of the given parity; false if it has not
// completed within about a second (the caller reports SEQ_STALLED).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity) {
  const unsigned long long t0 = global_ns();
  for (;;) {
    uint32_t ok;
    asm volatile("{\n\t.reg .pred p;\n\tmbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
                 "selp.u32 %0, 1, 0, p;\n\t}"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    if (ok) return true;
    if (global_ns() - t0 > 1000000000ull) return false;
  }
}
__device__ __forceinline__ void grid_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
// cp.async of 16 bytes to a shared-window address; 16-byte shared load.
__device__ __forceinline__ void cp_async16_to(uint32_t saddr, const void* gmem) {
  asm volatile("cp.async.cg.shared.global.L2::256B [%0], [%1], 16;" ::"r"(saddr), "l"(gmem) : "memory");
}
__device__ __forceinline__ uint4 lds128(uint32_t saddr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(saddr) : "memory");
  return v;
}

// ---------------------------------------------------------------- warp helpers
__device__ __forceinline__ unsigned lanemask_lt() {
  unsigned m;
  asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
  return m;
}
__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
  const uint32_t lo = __shfl_sync(kFull, static_cast<uint32_t>(v), src);
  const uint32_t hi = __shfl_sync(kFull, static_cast<uint32_t>(v >> 32), src);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t shfl_xor_u64(uint64_t v, int m) {
  const uint32_t lo = __shfl_xor_sync(kFull, static_cast<uint32_t>(v), m);
  const uint32_t hi = __shfl_xor_sync(kFull, static_cast<uint32_t>(v >> 32), m);
  return (static_cast<uint64_t>(hi) << 32) | lo;
}
__device__ __forceinline__ uint64_t warp_max_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
    const uint64_t t = shfl_xor_u64(v, o);
    v = t > v ? t : v;
  }
  return v;
}
__device__ __forceinline__ double warp_sum_f64(double v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
  return v;
}
__device__ __forceinline__ double warp_incl_scan_f64(double v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const double t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  return v;
}
__device__ __forceinline__ uint32_t warp_incl_scan_u32(uint32_t v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t t = __shfl_up_sync(kFull, v, o);
    if (lane >= o) v += t;
  }
  return v;
}

}  // namespace sv

namespace sv {

// ---------------------------------------------------------------- warp sort
// Bitonic sort of 128 64-bit keys held 4 per lane in blocked layout (lane l
// holds positions 4l..4l+3), into descending order.  Pad with 0 to sort fewer.
__device__ __forceinline__ void warp_sort128_desc(uint64_t (&v)[4], int lane) {
#pragma unroll
  for (int size = 2; size <= 128; size <<= 1) {
#pragma unroll
    for (int stride = size >> 1; stride > 0; stride >>= 1) {
      if (stride >= 4) {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const int i = 4 * lane + j;
          const uint64_t o = shfl_xor_u64(v[j], stride >> 2);
          const bool desc = (i & size) == 0;           // this block ends up descending
          const bool lower = (i & stride) == 0;        // lower position of the pair
          const bool keep_max = lower == desc;
          v[j] = keep_max ? (o > v[j] ? o : v[j]) : (o < v[j] ? o : v[j]);
        }
      } else {
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          if ((j & stride) == 0) {
            const int jj = j | stride;
            const bool desc = ((4 * lane + j) & size) == 0;
            const uint64_t a = v[j], b = v[jj];
            const uint64_t hi = a > b ? a : b, lo = a > b ? b : a;
            v[j] = desc ? hi : lo;
            v[jj] = desc ? lo : hi;
          }
        }
      }
    }
  }
}

// ---------------------------------------------------------------- double-float
// A value carried as hi + lo (two floats), added with Knuth's two-sum: about
// 48 significant bits with float-pipe latency only.
struct df { float hi, lo; };
__device__ __forceinline__ df df_from(float x) { return {x, 0.0f}; }
__device__ __forceinline__ df df_add(df a, df b) {
  const float s = a.hi + b.hi;
  const float bb = s - a.hi;
  float e = (a.hi - (s - bb)) + (b.hi - bb);
  e += a.lo + b.lo;
  const float hi = s + e;
  return {hi, e - (hi - s)};
}
__device__ __forceinline__ double df_to_double(df a) { return static_cast<double>(a.hi) + static_cast<double>(a.lo); }
__device__ __forceinline__ df df_shfl_up(df a, int o) {
  return {__shfl_up_sync(kFull, a.hi, o), __shfl_up_sync(kFull, a.lo, o)};
}
__device__ __forceinline__ df df_shfl_xor(df a, int m) {
  return {__shfl_xor_sync(kFull, a.hi, m), __shfl_xor_sync(kFull, a.lo, m)};
}
__device__ __forceinline__ df df_shfl(df a, int src) {
  return {__shfl_sync(kFull, a.hi, src), __shfl_sync(kFull, a.lo, src)};
}
__device__ __forceinline__ df warp_incl_scan_df(df v, int lane) {
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const df t = df_shfl_up(v, o);
    if (lane >= o) v = df_add(v, t);
  }
  return v;
}
__device__ __forceinline__ df warp_sum_df(df v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = df_add(v, df_shfl_xor(v, o));
  return v;
}
// a >= b for double-float values (compares the exact sums' signs via df_add).
__device__ __forceinline__ bool df_ge(df a, df b) {
  const df d = df_add(a, {-b.hi, -b.lo});
  return d.hi > 0.0f || (d.hi == 0.0f && d.lo >= 0.0f);
}

}  // namespace sv
