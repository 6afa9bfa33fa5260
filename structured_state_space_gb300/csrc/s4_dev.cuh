// Device building blocks shared by the libs4 kernels: complex helpers,
// device status bits, register-resident small DFTs and Stockham FFT passes
// over a row held in (padded) shared memory.
//
// Transform conventions follow "Recurrent, LSTM, and structured state-space
// models", section "Radix-two discrete Fourier transform": forward
// ahat_k = sum_j a_j w^{jk} with w = exp(-2 pi i/M); the inverse uses conj(w)
// and the 1/M factor, which the callers apply.
#pragma once
#include <cuda_runtime.h>
#include <stdint.h>

#include "s4_internal.h"

namespace s4dev {

// ---- device status bits (kept in the first word of the workspace) ----------
constexpr unsigned ST_RES_DIAG = 1u;   // s(z_k) - lambda_j == 0 (fp32)
constexpr unsigned ST_RES_CORR = 2u;   // W(z_k) singular
constexpr unsigned ST_NONFINITE = 4u;  // non-finite root value or spectrum
constexpr unsigned ST_BAD_STEP = 8u;   // Delta <= 0 or not finite
constexpr unsigned ST_SINGULAR = 16u;  // G = I - (Delta/2) A not solved (zero d_j or singular W)
constexpr unsigned ST_STALL = 32u;     // a bounded wait on an asynchronous copy ran out

// ---- bounds-checked build -------------------------------------------------------
// With -DS4_BOUNDS_CHECK (a separate library, built for tests) every global and
// shared-memory index of the instrumented kernels is compared with the extent of
// its buffer; an index outside it is counted in this translation unit's device
// counter and the access is skipped (a load gives zero).  No trap: the counter is
// read by the host (s4_bounds_violations) after the kernels ran.  In the normal
// build S4_IN is `true` and the helpers are plain accesses.
#ifdef S4_BOUNDS_CHECK
static __device__ unsigned long long g_s4_oob;
static __device__ __noinline__ void s4_oob_hit() { atomicAdd(&g_s4_oob, 1ull); }
static __device__ __forceinline__ bool s4_in(long long i, long long n) {
  const bool ok = i >= 0 && i < n;
  if (!ok) s4_oob_hit();
  return ok;
}
#define S4_IN(i, n) ::s4dev::s4_in((long long)(i), (long long)(n))
// host side: this translation unit's counter (defines a function `name`)
#define S4_OOB_COUNTER(name)                                                   \
  unsigned long long name() {                                                  \
    unsigned long long v = 0;                                                  \
    if (cudaMemcpyFromSymbol(&v, ::s4dev::g_s4_oob, sizeof(v)) != cudaSuccess) \
      return ~0ull;                                                            \
    return v;                                                                  \
  }
#else
#define S4_IN(i, n) true
#endif

// checked loads and stores: p[i] with 0 <= i < n
template <typename T>
__device__ __forceinline__ T ld_chk(const T* p, long long i, long long n) {
  return S4_IN(i, n) ? p[i] : T{};
}
template <typename T>
__device__ __forceinline__ void st_chk(T* p, long long i, long long n, T v) {
  if (S4_IN(i, n)) p[i] = v;
}

// ---- complex helpers ----------------------------------------------------------
__device__ __forceinline__ float2 cadd(float2 a, float2 b) { return make_float2(a.x + b.x, a.y + b.y); }
__device__ __forceinline__ float2 csub(float2 a, float2 b) { return make_float2(a.x - b.x, a.y - b.y); }
__device__ __forceinline__ float2 cmul(float2 a, float2 b) {
  return make_float2(fmaf(a.x, b.x, -a.y * b.y), fmaf(a.x, b.y, a.y * b.x));
}
__device__ __forceinline__ float2 cscale(float2 a, float s) { return make_float2(a.x * s, a.y * s); }
__device__ __forceinline__ bool cfinite(float2 a) { return isfinite(a.x) && isfinite(a.y); }

// Spectra of the two real rows of z = u_b + i u_{b+1} from Z[k] and zp =
// Z[n-k], times the kernel spectrum kv: 2 U_b kv and 2 U_{b+1} kv, with
// U_b = (Z[k] + conj Z[n-k])/2 and U_{b+1} = (Z[k] - conj Z[n-k])/(2i).
__device__ __forceinline__ void split_mul(float2 zk, float2 zp, float2 kv, float2& a0, float2& a1) {
  a0 = cmul(make_float2(zk.x + zp.x, zk.y - zp.y), kv);
  a1 = cmul(make_float2(zk.y + zp.y, zp.x - zk.x), kv);
}

// Approximate reciprocal (PTX rcp.approx.ftz.f32, relative error ~2^-23).
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

// ---- programmatic dependent launch --------------------------------------------------
// A kernel launched with the programmatic-serialization attribute may start
// while the previous kernel on the stream is still running; it must call
// pdl_wait() before it reads anything that kernel writes (a no-op for a
// normal launch).  pdl_launch_dependents() lets the next such kernel start.
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// ---- device status of a call (see St) --------------------------------------------
using s4impl::St;

// Set `flags` for this call: the 64-bit word (flags, generation) takes this
// call's generation, keeping the flags already set in it only if they carry
// the same generation.  A CAS loop; every failed round means another thread's
// update went in, and the loop is bounded all the same.
__device__ __forceinline__ void st_flag(St st, unsigned flags) {
  unsigned long long* w = reinterpret_cast<unsigned long long*>(st.w);
  unsigned long long old = *reinterpret_cast<volatile unsigned long long*>(w);
  for (int it = 0; it < (1 << 16); ++it) {
    const unsigned base = (unsigned)(old >> 32) == st.gen ? (unsigned)old : 0u;
    const unsigned long long nw = ((unsigned long long)st.gen << 32) | base | flags;
    if (nw == old) return;
    const unsigned long long prev = atomicCAS(w, old, nw);
    if (prev == old) return;
    old = prev;
  }
}
// Whether a kernel of this call has set a flag so far.
__device__ __forceinline__ bool st_bad(St st) {
  const unsigned long long v = *reinterpret_cast<volatile const unsigned long long*>(st.w);
  return (unsigned)(v >> 32) == st.gen && (unsigned)v != 0u;
}
// The first kernel of a call records its generation for s4_get_status.
__device__ __forceinline__ void st_record_gen(St st) {
  if (blockIdx.x == 0 && blockIdx.y == 0 && blockIdx.z == 0 && threadIdx.x == 0) st.w[2] = st.gen;
}

// Hint: bring the line holding p into L2 (no effect on results).
__device__ __forceinline__ void prefetch_l2(const void* p) {
  asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

// ---- bulk asynchronous copies into shared memory, tracked by an mbarrier -----------
// One thread announces the bytes of a round (mbar_expect_tx) and issues the
// copies (bulk_g2s: 16-byte aligned addresses, sizes a multiple of 16); every
// thread then waits for the round's phase.  The wait is bounded: it reports
// false after `limit` polls (kMbarWaitLimit unless the library's wait limit
// was changed, see s4_set_wait_limit) instead of spinning forever.
//
// Drain rule for a kernel whose wait gave up: the copy round it waited for
// may still be writing into shared memory.  The CTA then issues no further
// copies, reads what it would have staged straight from global memory, and
// before it exits waits once more, with the default limit, for that round.
constexpr int kMbarWaitLimit = 1 << 22;
__device__ __forceinline__ unsigned smem_u32(const void* p) {
  return (unsigned)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(unsigned long long* bar, unsigned count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
// make an initialised mbarrier visible to the asynchronous (copy) proxy
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// order this CTA's earlier shared-memory accesses before later asynchronous copies
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(unsigned long long* bar, unsigned bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, unsigned bytes, unsigned long long* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(smem_u32(dst)), "l"(src), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ bool mbar_wait(unsigned long long* bar, unsigned parity, int limit = kMbarWaitLimit) {
  for (int it = 0; it < limit; ++it) {
    unsigned done;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(done)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    if (done) return true;
  }
  return false;
}

// ---- padded shared-memory index: one spare slot per 16 entries ------------------
// Keeps the Stockham read (stride n/R) and write (stride p) patterns free of
// shared-memory bank conflicts for the radix plans used here.
__device__ __forceinline__ int pad(int w) { return w + (w >> 4); }
__host__ __device__ constexpr int padded_len(int n) { return n + (n >> 4) + 1; }

// ---- cos/sin of 2 pi e / 32 ----------------------------------------------------------
__host__ __device__ constexpr float cos32(int e) {
  // cos(k pi/16), k = 0..8, and the symmetries of the cosine
  constexpr float c[9] = {1.f,
                          0.98078528040323044f,
                          0.92387953251128674f,
                          0.83146961230254524f,
                          0.70710678118654752f,
                          0.55557023301960222f,
                          0.38268343236508978f,
                          0.19509032201612826f,
                          0.f};
  e &= 31;
  return e <= 8 ? c[e] : e <= 16 ? -c[16 - e] : e <= 24 ? -c[e - 16] : c[32 - e];
}
__host__ __device__ constexpr float sin32(int e) { return cos32(e - 8); }  // sin x = cos(x - pi/2)

// a <- a + w b, b <- a - w b, with w = exp(-+ 2 pi i e/32) (forward / inverse).
template <bool INV>
__device__ __forceinline__ void bfly(float2& a, float2& b, int e) {
  if (e == 0) {
    const float2 t = b;
    b = csub(a, t);
    a = cadd(a, t);
  } else if (e == 8) {  // w = -i (forward) or +i (inverse)
    const float2 t = INV ? make_float2(-b.y, b.x) : make_float2(b.y, -b.x);
    b = csub(a, t);
    a = cadd(a, t);
  } else {
    const float c = cos32(e);
    const float s = INV ? sin32(e) : -sin32(e);  // w = c + i s
    const float yx = fmaf(b.x, c, fmaf(-b.y, s, a.x));
    const float yy = fmaf(b.x, s, fmaf(b.y, c, a.y));
    b = make_float2(fmaf(2.f, a.x, -yx), fmaf(2.f, a.y, -yy));
    a = make_float2(yx, yy);
  }
}

// Same butterfly when only a + w b is wanted.
template <bool INV>
__device__ __forceinline__ void bfly_top(float2& a, const float2 b, int e) {
  if (e == 0) {
    a = cadd(a, b);
  } else if (e == 8) {
    a = cadd(a, INV ? make_float2(-b.y, b.x) : make_float2(b.y, -b.x));
  } else {
    const float c = cos32(e);
    const float s = INV ? sin32(e) : -sin32(e);
    a = make_float2(fmaf(b.x, c, fmaf(-b.y, s, a.x)), fmaf(b.x, s, fmaf(b.y, c, a.y)));
  }
}

// In-register DFT of length R (1, 2, 4, 8, 16, 32) by the even/odd split of the
// radix-two recursion.  HALFZERO: inputs R/2..R-1 are known zero.  HALFOUT:
// only outputs 0..R/2-1 are needed.
template <int R, bool INV, bool HALFZERO = false, bool HALFOUT = false>
__device__ __forceinline__ void dft(float2* a) {
  if constexpr (R == 1) {
    return;
  } else if constexpr (R == 2) {
    if constexpr (HALFZERO) {
      a[1] = a[0];
    } else if constexpr (HALFOUT) {
      a[0] = cadd(a[0], a[1]);
    } else {
      bfly<INV>(a[0], a[1], 0);
    }
  } else {
    float2 ev[R / 2], od[R / 2];
#pragma unroll
    for (int j = 0; j < R / 2; ++j) {
      ev[j] = a[2 * j];
      od[j] = a[2 * j + 1];
    }
    dft<R / 2, INV, HALFZERO>(ev);
    dft<R / 2, INV, HALFZERO>(od);
#pragma unroll
    for (int k = 0; k < R / 2; ++k) {
      if constexpr (HALFOUT) {
        bfly_top<INV>(ev[k], od[k], (32 / R) * k);
        a[k] = ev[k];
      } else {
        bfly<INV>(ev[k], od[k], (32 / R) * k);
        a[k] = ev[k];
        a[k + R / 2] = od[k];
      }
    }
  }
}

__host__ __device__ constexpr int highbit(int q) {
  int h = 1;
  while (h * 2 <= q) h *= 2;
  return h;
}

// a[q] *= w^q, q = 1..R-1 (w already conjugated for an inverse pass).
template <int R>
__device__ __forceinline__ void apply_twiddles(float2* a, float2 w) {
  if constexpr (R > 1) {
    float2 pw[R];
    pw[1] = w;
#pragma unroll
    for (int q = 2; q < R; ++q) {
      const int hb = highbit(q);
      pw[q] = (hb == q) ? cmul(pw[q / 2], pw[q / 2]) : cmul(pw[hb], pw[q - hb]);
    }
#pragma unroll
    for (int q = 1; q < R; ++q) a[q] = cmul(a[q], pw[q]);
  }
}

}  // namespace s4dev
