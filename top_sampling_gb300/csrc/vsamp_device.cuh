// Device helpers for the sampling-stage kernels (sm_103a): bulk-copy / mbarrier / cluster PTX
// wrappers, Philox4x32-10, order-preserving keys, fixed-point mass and reductions.
#pragma once

#include <cstdint>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cooperative_groups.h>

namespace vsamp {
namespace cg = cooperative_groups;

constexpr uint32_t kFullMask = 0xFFFFFFFFu;
// Fixed-point scale of probability mass: w in (0, 1] is stored as round(w * 2^40) in a uint64.
// A 2^21-token row sums to < 2^61, so row totals never overflow.
constexpr int kMassShift = 40;
constexpr float kMassScale = 1099511627776.0f;   // 2^40

// ------------------------------------------------------------------------------------------------
// Shared-memory addressing, bulk copies and mbarriers (PTX ISA: cp.async.bulk, mbarrier).
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(void* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(void* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

// Global -> own shared memory bulk copy; completion is signalled on `bar` as transaction bytes.
// dst, src and bytes must all be multiples of 16.
__device__ __forceinline__ void bulk_copy_g2s(void* dst, const void* src, uint32_t bytes, void* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst)),
      "l"(src), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Orders this thread's earlier generic-proxy accesses to shared memory before later async-proxy
// (bulk copy) writes to it.
__device__ __forceinline__ void fence_proxy_async_shared() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ bool mbar_try_wait(void* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Arrival on an mbarrier of another CTA of the cluster (a shared::cluster address from mapa), with
// release semantics at cluster scope: this thread's earlier writes to that CTA's shared memory are
// visible to whoever observes the completed phase.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

// Test of an mbarrier phase with acquire semantics at cluster scope (pairs with mbar_arrive_remote).
__device__ __forceinline__ bool mbar_try_wait_cluster(void* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

__device__ __forceinline__ bool mbar_wait_cluster_bounded(void* bar, uint32_t parity, long long max_cycles) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait_cluster(bar, parity)) return true;
    if (clock64() - t0 > max_cycles) return false;
  }
}

// Bounded wait on an mbarrier phase: gives up after ~`max_cycles` SM clock cycles and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(void* bar, uint32_t parity, long long max_cycles) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long t0 = clock64();
  for (;;) {
    for (int i = 0; i < 64; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (clock64() - t0 > max_cycles) return false;
  }
}

// Cluster-wide barrier of all threads that publishes this thread's earlier shared-memory writes to the
// peers (a release restricted to shared memory, so stores to global memory still in flight are not
// waited for) and acquires theirs. It also synchronises the threads of this CTA.
__device__ __forceinline__ void cluster_barrier_shared() {
  asm volatile("fence.release.sync_restrict::shared::cta.cluster;" ::: "memory");
  asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");
  asm volatile("barrier.cluster.wait.aligned;" ::: "memory");
}

// ------------------------------------------------------------------------------------------------
// Distributed shared memory: a CTA's shared address mapped into the address window of CTA `rank` of
// the cluster, stores and an acquire-release atomic add there.
// ------------------------------------------------------------------------------------------------
// Acquire-release add on a word of this CTA's shared memory, at CTA scope; returns the old value.
__device__ __forceinline__ uint32_t smem_atomic_add_acq_rel_cta(void* p, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cta.shared::cta.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(smem_addr(p)), "r"(v) : "memory");
  return old;
}

__device__ __forceinline__ uint32_t dsmem_map(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_addr(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void dsmem_store_v4(uint32_t addr, uint32_t a, uint32_t b, uint32_t c, uint32_t d) {
  asm volatile("st.shared::cluster.v4.u32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(a), "r"(b), "r"(c), "r"(d)
               : "memory");
}
// 16 bytes into a peer CTA's shared memory (addr mapped by dsmem_map) whose arrival is counted in bytes on the
// peer's mbarrier `bar` (mapped too): the issuing thread neither waits for the write nor orders its own earlier
// memory operations before it; the peer's wait on `bar` (acquire, cluster scope) makes the bytes visible.
__device__ __forceinline__ void dsmem_store_async_v4(uint32_t addr, uint4 v, uint32_t bar) {
  asm volatile("st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
               ::"r"(addr), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(bar)
               : "memory");
}
__device__ __forceinline__ uint4 dsmem_load_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr)
               : "memory");
  return v;
}
__device__ __forceinline__ unsigned long long dsmem_load_u64(uint32_t addr) {
  unsigned long long v;
  asm volatile("ld.shared::cluster.u64 %0, [%1];" : "=l"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t dsmem_load_u32(uint32_t addr) {
  uint32_t v;
  asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ void dsmem_store_u32(uint32_t addr, uint32_t v) {
  asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
// Atomic add at cluster scope with acquire-release ordering; returns the previous value.
__device__ __forceinline__ uint32_t dsmem_atomic_add_acq_rel(uint32_t addr, uint32_t v) {
  uint32_t old;
  asm volatile("atom.acq_rel.cluster.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
  return old;
}

// ------------------------------------------------------------------------------------------------
// Philox4x32-10 (Salmon, Moraes, Dror, Shaw, "Parallel Random Numbers: As Easy as 1, 2, 3", SC'11).
// Round: (c0,c1,c2,c3) -> (hi(M1*c2)^c1^k0, lo(M1*c2), hi(M0*c0)^c3^k1, lo(M0*c0)); the key advances by
// the Weyl constants between rounds.
// ------------------------------------------------------------------------------------------------
struct PhiloxKey {
  uint32_t k0, k1;
};

__device__ __forceinline__ uint4 philox4x32_10(uint4 c, PhiloxKey key) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
  constexpr uint32_t W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
  uint32_t k0 = key.k0, k1 = key.k1;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    // one 32x32 -> 64-bit product per multiplier, split into its high and low words
    unsigned long long p0, p1;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(c.x), "r"(M0));
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(c.z), "r"(M1));
    const uint32_t lo0 = (uint32_t)p0, hi0 = (uint32_t)(p0 >> 32);
    const uint32_t lo1 = (uint32_t)p1, hi1 = (uint32_t)(p1 >> 32);
    c = make_uint4(hi1 ^ c.y ^ k0, lo1, hi0 ^ c.w ^ k1, lo0);
    k0 += W0;
    k1 += W1;
  }
  return c;
}

// The ten round keys of a Philox4x32-10 key, computed once for many calls.
struct PhiloxRoundKeys {
  uint32_t k0[10], k1[10];
  __device__ __forceinline__ explicit PhiloxRoundKeys(PhiloxKey key) {
#pragma unroll
    for (int r = 0; r < 10; ++r) {
      k0[r] = key.k0 + (uint32_t)r * 0x9E3779B9u;
      k1[r] = key.k1 + (uint32_t)r * 0xBB67AE85u;
    }
  }
};

// Philox4x32-10 with precomputed round keys (same output as philox4x32_10).
__device__ __forceinline__ uint4 philox4x32_10_rk(uint4 c, const PhiloxRoundKeys& K) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    unsigned long long p0, p1;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(c.x), "r"(M0));
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(c.z), "r"(M1));
    const uint32_t lo0 = (uint32_t)p0, hi0 = (uint32_t)(p0 >> 32);
    const uint32_t lo1 = (uint32_t)p1, hi1 = (uint32_t)(p1 >> 32);
    c = make_uint4(hi1 ^ c.y ^ K.k0[r], lo1, hi0 ^ c.w ^ K.k1[r], lo0);
  }
  return c;
}

// Philox4x32-10 along one row: the counters (c0, c1, c2, c3) of a row differ only in c0, so the first
// round's product M1 * c2 and the second round's product M0 * x1 (x1, y1: the first round's output words
// that do not depend on c0) are formed once. Each counter then costs 18 wide multiplies instead of 20.
// Same output as philox4x32_10.
struct PhiloxRow {
  uint32_t k0[10], k1[10];   // round keys
  uint32_t y1, z1k;          // first round: y1 = lo(M1 c2); z1k = c3 ^ k1[0]
  uint32_t x2k, hi2, w2;     // second round: x2k = y1 ^ k0[1]; hi2 ^ ..., w2 = hi / lo of M0 * x1
  __device__ __forceinline__ PhiloxRow(PhiloxKey key, uint32_t c1, uint32_t c2, uint32_t c3) {
    constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
#pragma unroll
    for (int r = 0; r < 10; ++r) {
      k0[r] = key.k0 + (uint32_t)r * 0x9E3779B9u;
      k1[r] = key.k1 + (uint32_t)r * 0xBB67AE85u;
    }
    const unsigned long long p1 = (unsigned long long)M1 * c2;
    const uint32_t x1 = (uint32_t)(p1 >> 32) ^ c1 ^ k0[0];
    y1 = (uint32_t)p1;
    z1k = c3 ^ k1[0];
    const unsigned long long p2 = (unsigned long long)M0 * x1;
    x2k = y1 ^ k0[1];
    hi2 = (uint32_t)(p2 >> 32) ^ k1[1];
    w2 = (uint32_t)p2;
  }
  __device__ __forceinline__ uint4 operator()(uint32_t c0) const {
    constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u;
    unsigned long long p0, p1;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(c0), "r"(M0));
    const uint32_t z1 = (uint32_t)(p0 >> 32) ^ z1k, w1 = (uint32_t)p0;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(z1), "r"(M1));
    uint4 c = make_uint4((uint32_t)(p1 >> 32) ^ x2k, (uint32_t)p1, hi2 ^ w1, w2);
#pragma unroll
    for (int r = 2; r < 10; ++r) {
      asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(c.x), "r"(M0));
      asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(c.z), "r"(M1));
      c = make_uint4((uint32_t)(p1 >> 32) ^ c.y ^ k0[r], (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c.w ^ k1[r],
                     (uint32_t)p0);
    }
    return c;
  }
};

__device__ __forceinline__ uint32_t min4_u32(uint4 w) { return min(__vimin3_u32(w.x, w.y, w.z), w.w); }

// 4-bit draw code of a 16-byte vector from the smallest Philox word w of its tokens: min(clz(w), 15).
// w < bk implies code(w) >= code(bk), so testing codes flags a superset of the vectors the prune bound keeps.
__device__ __forceinline__ uint32_t draw_code(uint32_t w) { return min((uint32_t)__clz(w), 15u); }


// PhiloxRow with few live registers: the round keys from the third round on are formed as the rounds run
// (one add per key word and round, shared by the counters drawn together), and only the smallest of each
// counter's four output words is returned. Same words as philox4x32_10.
struct PhiloxRowMin {
  uint32_t k0_2, k1_2;       // round keys of the third round
  uint32_t y1, z1k, x2k, hi2, w2;
  __device__ __forceinline__ PhiloxRowMin(PhiloxKey key, uint32_t c1, uint32_t c2, uint32_t c3) {
    constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u, W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    const unsigned long long p1 = (unsigned long long)M1 * c2;
    const uint32_t x1 = (uint32_t)(p1 >> 32) ^ c1 ^ key.k0;
    y1 = (uint32_t)p1;
    z1k = c3 ^ key.k1;
    const unsigned long long p2 = (unsigned long long)M0 * x1;
    x2k = y1 ^ (key.k0 + W0);
    hi2 = (uint32_t)(p2 >> 32) ^ (key.k1 + W1);
    w2 = (uint32_t)p2;
    k0_2 = key.k0 + 2u * W0;
    k1_2 = key.k1 + 2u * W1;
  }
  // the smallest output word of each of N counters
  template <int N>
  __device__ __forceinline__ void min_words(const uint32_t (&c0)[N], uint32_t (&m)[N]) const {
    constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u, W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
    uint4 c[N];
#pragma unroll
    for (int n = 0; n < N; ++n) {
      unsigned long long p0, p1;
      asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(c0[n]), "r"(M0));
      const uint32_t z1 = (uint32_t)(p0 >> 32) ^ z1k, w1 = (uint32_t)p0;
      asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(z1), "r"(M1));
      c[n] = make_uint4((uint32_t)(p1 >> 32) ^ x2k, (uint32_t)p1, hi2 ^ w1, w2);
    }
    uint32_t k0 = k0_2, k1 = k1_2;
#pragma unroll
    for (int r = 2; r < 10; ++r) {
#pragma unroll
      for (int n = 0; n < N; ++n) {
        unsigned long long p0, p1;
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(c[n].x), "r"(M0));
        asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(c[n].z), "r"(M1));
        c[n] = make_uint4((uint32_t)(p1 >> 32) ^ c[n].y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ c[n].w ^ k1,
                          (uint32_t)p0);
      }
      k0 += W0;
      k1 += W1;
    }
#pragma unroll
    for (int n = 0; n < N; ++n) m[n] = min4_u32(c[n]);
  }
};

// PhiloxRowMin's rounds returning all four output words of each of N counters (same words as philox4x32_10).
template <int N>
__device__ __forceinline__ void philox_row_words(const PhiloxRowMin& ph, const uint32_t (&c0)[N], uint4 (&out)[N]) {
  constexpr uint32_t M0 = 0xD2511F53u, M1 = 0xCD9E8D57u, W0 = 0x9E3779B9u, W1 = 0xBB67AE85u;
#pragma unroll
  for (int n = 0; n < N; ++n) {
    unsigned long long p0, p1;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(c0[n]), "r"(M0));
    const uint32_t z1 = (uint32_t)(p0 >> 32) ^ ph.z1k, w1 = (uint32_t)p0;
    asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(z1), "r"(M1));
    out[n] = make_uint4((uint32_t)(p1 >> 32) ^ ph.x2k, (uint32_t)p1, ph.hi2 ^ w1, ph.w2);
  }
  uint32_t k0 = ph.k0_2, k1 = ph.k1_2;
#pragma unroll
  for (int r = 2; r < 10; ++r) {
#pragma unroll
    for (int n = 0; n < N; ++n) {
      unsigned long long p0, p1;
      asm("mul.wide.u32 %0, %1, %2;" : "=l"(p0) : "r"(out[n].x), "r"(M0));
      asm("mul.wide.u32 %0, %1, %2;" : "=l"(p1) : "r"(out[n].z), "r"(M1));
      out[n] = make_uint4((uint32_t)(p1 >> 32) ^ out[n].y ^ k0, (uint32_t)p1, (uint32_t)(p0 >> 32) ^ out[n].w ^ k1,
                          (uint32_t)p0);
    }
    k0 += W0;
    k1 += W1;
  }
}

__device__ __forceinline__ uint32_t philox_word(uint4 w, int lane) {
  return lane == 0 ? w.x : lane == 1 ? w.y : lane == 2 ? w.z : w.w;
}

// ------------------------------------------------------------------------------------------------
// Order-preserving keys. fp32: positive -> bits | 0x80000000, negative -> ~bits; -0.0 reads as +0.0.
// bf16 uses the same map on 16 bits. key32_of_key16 widens a bf16 key to the fp32 key of the same value.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ uint32_t key_f32_bits(uint32_t b) {
  b = (b == 0x80000000u) ? 0u : b;
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}
__device__ __forceinline__ uint32_t key_bf16_bits(uint32_t h) {
  h &= 0xFFFFu;
  h = (h == 0x8000u) ? 0u : h;
  return (h & 0x8000u) ? (~h & 0xFFFFu) : (h | 0x8000u);
}
__device__ __forceinline__ uint32_t key32_of_key16(uint32_t k16) {
  return (k16 << 16) | ((k16 & 0x8000u) ? 0u : 0xFFFFu);
}
__device__ __forceinline__ float value_of_key32(uint32_t k) {
  const uint32_t b = (k & 0x80000000u) ? (k ^ 0x80000000u) : ~k;
  return __uint_as_float(b);
}

// ------------------------------------------------------------------------------------------------
// exp as 2^(s * log2 e) with the hardware ex2 approximation (relative error of a few ulp). Results
// below 2^-126 flush to zero: every caller either rounds them to zero anyway (2^-40 fixed-point masses)
// or uses them in a prune test where a token that small can never be drawn.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float ex2_approx(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;

// round(w * 2^40), ties to even, for 0 <= w < 16, without a 64-bit conversion instruction (those run on the
// FP64 pipe, a few results per clock per SM on this part): v = w * 2^40 < 2^44 is split into h (v rounded
// at the granularity 2^21) and l = v - h (exact, |l| <= 2^20); each becomes an integer by adding a power of
// two that puts the unit in the last mantissa bit. The sum is v rounded to nearest-even because h is even.
__device__ __forceinline__ uint64_t mass_fx(float w) {
  const float v = w * kMassScale;
  const float big = 26388279066624.0f;          // 1.5 * 2^44: unit in the last place 2^21
  const float h = (v + big) - big;
  const float l = v - h;
  const uint32_t hi = __float_as_uint(fmaf(h, 4.76837158203125e-07f, 8388608.0f)) - 0x4B000000u;   // h / 2^21
  const int32_t lo = (int32_t)(__float_as_uint(l + 12582912.0f) - 0x4B400000u);                   // round(l)
  return ((uint64_t)hi << 21) + (uint64_t)(int64_t)lo;
}

// ceil(p * S) for an fp32 p in [0, 1] and a fixed-point mass S < 2^63, exactly, in integer arithmetic:
// p = m * 2^(e - 150) with a 24-bit m, and the 88-bit product m * S is shifted right with rounding up.
__host__ __device__ __forceinline__ unsigned long long ceil_mul_frac(float p, unsigned long long S) {
  if (!(p > 0.f)) return 0ull;
  if (p >= 1.f) return S;
#ifdef __CUDA_ARCH__
  const uint32_t bits = __float_as_uint(p);
#else
  uint32_t bits;
  __builtin_memcpy(&bits, &p, 4);
#endif
  uint32_t e = (bits >> 23) & 0xFFu;
  unsigned long long m = bits & 0x7FFFFFu;
  if (e) m |= 0x800000u; else e = 1;
  const int sh = 150 - (int)e;                      // >= 24 because p < 1
  const unsigned long long lo = m * S;
#ifdef __CUDA_ARCH__
  const unsigned long long hi = __umul64hi(m, S);
#else
  const unsigned long long hi = (unsigned long long)(((unsigned __int128)m * S) >> 64);
#endif
  unsigned long long qv;
  bool rem;
  if (sh < 64) {
    qv = (lo >> sh) | (hi << (64 - sh));
    rem = (lo & ((1ull << sh) - 1ull)) != 0ull;
  } else if (sh == 64) {
    qv = hi;
    rem = lo != 0ull;
  } else if (sh < 128) {
    qv = hi >> (sh - 64);
    rem = lo != 0ull || (hi & ((1ull << (sh - 64)) - 1ull)) != 0ull;
  } else {
    qv = 0ull;
    rem = (lo | hi) != 0ull;
  }
  return qv + (rem ? 1ull : 0ull);
}

// A 64-bit count or fixed-point mass as fp32 (two exact 32-bit conversions, relative error ~1e-7).
__device__ __forceinline__ float u64_to_float(unsigned long long v) {
  return fmaf((float)(uint32_t)(v >> 32), 4294967296.0f, (float)(uint32_t)v);
}

// ------------------------------------------------------------------------------------------------
// Warp reductions.
// ------------------------------------------------------------------------------------------------
__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFullMask, v, o));
  return v;
}
__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) v += __shfl_xor_sync(kFullMask, v, o);
  return v;
}
__device__ __forceinline__ uint32_t warp_sum_u32(uint32_t v) { return __reduce_add_sync(kFullMask, v); }
__device__ __forceinline__ uint32_t warp_max_u32(uint32_t v) { return __reduce_max_sync(kFullMask, v); }
__device__ __forceinline__ uint32_t warp_min_u32(uint32_t v) { return __reduce_min_sync(kFullMask, v); }

// (score, index) arg-max with ties to the lower index.
struct ArgMax {
  float score;
  int32_t idx;
  float s;        // max-subtracted, temperature-scaled logit of idx
};
__device__ __forceinline__ bool argmax_better(float a, int32_t ia, float b, int32_t ib) {
  return a > b || (a == b && ia < ib);
}
__device__ __forceinline__ ArgMax warp_argmax(ArgMax v) {
#pragma unroll
  for (int o = 16; o; o >>= 1) {
    ArgMax w;
    w.score = __shfl_xor_sync(kFullMask, v.score, o);
    w.idx = __shfl_xor_sync(kFullMask, v.idx, o);
    w.s = __shfl_xor_sync(kFullMask, v.s, o);
    if (argmax_better(w.score, w.idx, v.score, v.idx)) v = w;
  }
  return v;
}

}  // namespace vsamp
