// The sampling kernel with specialised warps (vsamp_sample).
//
// One thread-block cluster of C CTAs owns a row, as in the row engine: each CTA holds a slice of the row in
// shared memory, bulk-copied from HBM once. Each CTA has kDataWarps data warps and one control warp:
//   data warps    stream the slice: P1 (maximum, non-finite check), P2 (fixed-point mass, maxima, min-p
//                 statistics), radix histogram and tie-count passes on request, the cut's boundary, and
//                 P4 (Philox4x32-10 Gumbel-max over the kept prefix). Each warp copies the next row into its
//                 region of the slice as soon as it has finished the row.
//   control warp  takes every per-row decision from the data warps' partials: the cluster exchanges
//                 (each CTA's message written into every peer's shared memory, counted on an mbarrier),
//                 the top-k / top-p / min-p plan and radix rounds, the prune bound of the draw, the
//                 cluster arg-max and the row's outputs.
// The two hand over through named barriers (data -> control: bar.arrive / bar.sync, and back), so data
// warps never wait on a cluster barrier, carry little state through their loops, and the per-row scalar
// work runs once per CTA instead of once per warp.
//
// The arithmetic is that of the row engine (vsamp_row.cuh) and gives the same results: masses in 2^-40
// fixed point summed per 16-byte vector in a fixed order, cuts found by the same rules, the same Philox
// counters and prune bound.
#pragma once

#include <cstddef>

#include "vsamp_row.cuh"

namespace vsamp {

constexpr int kMaxDataWarps = 8;

// named barriers (0 is __syncthreads)
enum SampleBarrier : int { SB_P1 = 1, SB_CTL = 2, SB_P2 = 3, SB_HIST = 4, SB_P4 = 5 };
// control -> data requests after P2
enum SampleRequest : int { REQ_DONE = 0, REQ_HIST = 1, REQ_COUNT = 2, REQ_ABORT = 3, REQ_MASS = 4, REQ_GATHER = 5 };
// how the data warps find the cut's last kept element
enum CutGroup : int {
  GROUP_MAX = 0,     // inside the maxima: counts and prefixes from P2
  GROUP_PIVOT = 1,   // inside the pivot value's group: counts from a tie-count pass
  GROUP_WHOLE = 2,   // the pivot group is kept whole: x >= xP
  GROUP_ALL = 3,     // every element
};

// named barrier over all nthreads threads of the CTA (a multiple of 32)
__device__ __forceinline__ void nb_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
__device__ __forceinline__ void nb_arrive(int id, int nthreads) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

// Control -> data message (written by the control warp before it arrives on SB_CTL).
struct SampleCtl {
  int32_t status;
  int32_t req;
  int32_t group;
  int32_t one_token;        // greedy, or the cut keeps one token
  int32_t all_cand;         // every kept token is a draw candidate
  int32_t minp_on;
  int32_t hist_mass;        // REQ_HIST: also histogram masses
  int32_t hpar;             // REQ_HIST: histogram buffer
  int32_t shift;            // REQ_HIST: bin = (key >> shift) & 255 for keys matching prefix above shift + 8
  uint32_t prefix;           // REQ_HIST: the prefix; REQ_MASS: keys above it are summed
  uint32_t floor_rk;        // REQ_HIST: keys below it are left out
  int32_t hfirst;           // REQ_HIST: the first round of a search (every vector is visited)
  int32_t kfloor;           // REQ_HIST, REQ_COUNT: only keys at or above the top-k pivot of the last REQ_MASS
                            // matter (the first round, or the count, visits only the vectors holding one)
  int32_t vround;           // REQ_HIST: bins are value bins (vxlo, vsc) instead of key bytes
  int32_t vsel;             // REQ_HIST key round after a value round, REQ_MASS after a count search: the value
                            // bin the search's value round selected (only vectors whose largest bin is at or
                            // above it are visited); -1: none
  int32_t p4km;             // the draw visits only the vectors holding a key at or above the top-k pivot
  float vxlo, vsc;
  uint32_t klo, khi;        // REQ_HIST key rounds: only keys in [klo, khi] (the selected value bin)
  uint32_t kmin32;          // min-p threshold (fp32 key space)
  uint32_t bk;              // prune bound on the Philox word
  uint32_t rid, st_lo, st_hi, k0, k1;
  float M, c1, invT, xP, kappa;
  unsigned long long need;  // elements of the cut group that are kept
  uint32_t wstart[kMaxDataWarps];   // elements of the cut group before each data warp's chunk (whole row)
};

struct SampleSmem {
  unsigned long long lbar[2][kMaxDataWarps];   // per slice buffer and data warp: its region has landed
  unsigned long long xbar[2];            // cluster exchange: the local arrival and the C messages' bytes, per parity
  uint4 xm[2][16][2];                    // cluster exchange mailboxes: each CTA's 32-byte message
  uint4 dp[kMaxDataWarps][2];            // data -> control partials (P1, P2, tie counts)
  uint4 ap[kMaxDataWarps];               // P4 partials: score, index, scaled logit, boundary index
  uint4 aslot[2][16];                    // CTA 0's copy: each CTA's P4 partial, per row parity
  uint32_t acnt[2];                      // CTA 0's copy: CTAs that have published, per row parity
  SampleCtl ctl;
  __align__(16) uint32_t hcnt[2][256];   // radix histograms (count, mass low / high words), per round parity;
  __align__(16) unsigned long long hm[2][256];   // 16-byte aligned: read as 16-byte vectors
};

static_assert(offsetof(SampleSmem, hcnt) % 16 == 0 && offsetof(SampleSmem, hm) % 16 == 0,
              "the histograms are read as 16-byte vectors");

__host__ __device__ constexpr int sample_slice_offset() {
  return (int)((sizeof(SampleSmem) + 127) / 128 * 128);
}

// ------------------------------------------------------------------------------------------------
// Control warp: cluster exchange of one 32-byte message per CTA. Lane 0 arms this CTA's mbarrier for the
// C messages (C * 32 bytes, its own arrival the only one); lane r < C writes this CTA's message into CTA r's
// mailbox with two asynchronous 16-byte stores that count their bytes on CTA r's mbarrier, so the sender
// waits neither for the writes nor for its own earlier memory operations; lane 0 then waits (bounded) for
// this CTA's barrier. Afterwards every lane may read xm[par][0 .. C-1]. Returns false on timeout.
// Mailboxes are double-buffered by exchange parity: a CTA cannot reach exchange n + 2 before every peer
// has sent exchange n + 1, which each does only after reading exchange n. A peer's bytes may land before
// the local arming; the barrier's transaction count then runs below zero and the phase still cannot
// complete before the local arrival.
// ------------------------------------------------------------------------------------------------
struct ClusterXchg {
  int n = 0;   // exchanges so far
  __device__ __forceinline__ int par() const { return n & 1; }
  __device__ bool run(SampleSmem& sh, int C, int crank, uint4 m0, uint4 m1, long long wait_cycles) {
    const int lane = threadIdx.x & 31;
    const int pb = n & 1;
    const uint32_t ph = (uint32_t)((n >> 1) & 1);
    ++n;
    if (C == 1) {
      if (lane == 0) { sh.xm[pb][0][0] = m0; sh.xm[pb][0][1] = m1; }
      __syncwarp();
      return true;
    }
    if (lane == 0) mbar_arrive_expect_tx(&sh.xbar[pb], (uint32_t)(C * 32));
    if (lane < C) {
      const uint32_t dst = dsmem_map(&sh.xm[pb][crank][0], (uint32_t)lane);
      const uint32_t bar = dsmem_map(&sh.xbar[pb], (uint32_t)lane);
      dsmem_store_async_v4(dst, m0, bar);
      dsmem_store_async_v4(dst + 16u, m1, bar);
    }
    uint32_t ok = 1u;
    if (lane == 0) ok = mbar_wait_cluster_bounded(&sh.xbar[pb], ph, wait_cycles) ? 1u : 0u;
    ok = __shfl_sync(kFullMask, ok, 0);
    __syncwarp();
    return ok != 0u;
  }
};

__device__ __forceinline__ unsigned long long u64_of(uint32_t lo, uint32_t hi) {
  return ((unsigned long long)hi << 32) | lo;
}

// ------------------------------------------------------------------------------------------------
// Control warp: the draw over every kept token of a row (x > xP, or x == xP and index <= It), read from
// global memory, when the prune bound did not certify the cluster's winner. Out of line: it runs with
// probability ~1e-9 per row and would otherwise hold registers in the control warp's common path.
// ------------------------------------------------------------------------------------------------
template <typename T>
static __device__ __noinline__ ArgMax control_fallback_draw(const unsigned char* xrow, int64_t n, float xP, int32_t It,
                                                            float M, float invT, uint32_t rid, uint64_t st, uint64_t sd) {
  using Tr = Traits<T>;
  const int lane = threadIdx.x & 31;
  const PhiloxKey key{(uint32_t)sd, (uint32_t)(sd >> 32)};
  const uint32_t st_lo = (uint32_t)st, st_hi = (uint32_t)(st >> 32);
  float fs = -INFINITY, fsv = 0.f;
  int32_t fi = 0x7FFFFFFF;
  for (int64_t e = lane; e < n; e += 32) {
    const float xv = Tr::load_global(xrow, e);
    if (!(xv > xP || (xv == xP && e <= (int64_t)It))) continue;
    const uint4 w4 = philox4x32_10(make_uint4((uint32_t)(e >> 2), rid, st_lo, st_hi), key);
    const uint32_t bw = philox_word(w4, (int)(e & 3));
    const float sv = (xv - M) * invT;
    const float score = gumbel_score(sv, bw);
    if (argmax_better(score, (int32_t)e, fs, fi)) { fs = score; fi = (int32_t)e; fsv = sv; }
  }
  return warp_argmax(ArgMax{fs, fi, fsv});
}

// The vectors of a thread's chunk that hold a kept token, among the vectors vis (~0: every vector).
template <typename T>
static __device__ __noinline__ unsigned long long kept_vectors_in(const uint4* mine, int thr_n, int64_t thr_e0,
                                                                 float xP, int32_t It, unsigned long long vis) {
  if (vis == ~0ull) return kept_vectors<T>(mine, thr_n, thr_e0, xP, It);
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  const int nfull = thr_n / VE;
  unsigned long long m = 0ull;
  for (; vis; vis &= vis - 1ull) {
    const int j = __ffsll((long long)vis) - 1;
    float x[VE];
    Tr::values(mine[j], x);
    const int cnt = j < nfull ? VE : thr_n - nfull * VE;
    const int64_t e0 = thr_e0 + (int64_t)j * VE;
    bool any = false;
#pragma unroll
    for (int i = 0; i < VE; ++i) any |= i < cnt && (x[i] > xP || (x[i] == xP && e0 + i <= (int64_t)It));
    if (any) m |= 1ull << j;
  }
  return m;
}

// ------------------------------------------------------------------------------------------------
// P1 over one thread's vectors: the maximum, the minimum (mn_out; the first radix round bins values over
// the row's range), and nf != 0 when a value is NaN or +-inf (x * 0 is NaN exactly for those). bf16 pairs
// are handled packed.
// ------------------------------------------------------------------------------------------------
template <typename T>
static __device__ __noinline__ float max_pass(const uint4* mine, int thr_n, float& nf_out, float& mn_out) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  const int nfull = thr_n / VE;
  float mx = -INFINITY, mn = INFINITY, nf = 0.f;
  if constexpr (VE == 8) {
    const __nv_bfloat162 zero2 = __float2bfloat162_rn(0.f);
    __nv_bfloat162 mxa = __float2bfloat162_rn(-INFINITY), mxb = mxa, mna = __float2bfloat162_rn(INFINITY),
                   mnb = mna, nfa = zero2, nfb = zero2;
    for (int j = 0; j < nfull; ++j) {
      const uint4 v = mine[j];
      mxa = __hmax2(mxa, __hmax2(Tr::pair(v.x), Tr::pair(v.y)));
      mxb = __hmax2(mxb, __hmax2(Tr::pair(v.z), Tr::pair(v.w)));
      mna = __hmin2(mna, __hmin2(Tr::pair(v.x), Tr::pair(v.y)));
      mnb = __hmin2(mnb, __hmin2(Tr::pair(v.z), Tr::pair(v.w)));
      nfa = __hfma2(Tr::pair(v.x), zero2, __hfma2(Tr::pair(v.y), zero2, nfa));
      nfb = __hfma2(Tr::pair(v.z), zero2, __hfma2(Tr::pair(v.w), zero2, nfb));
    }
    mxa = __hmax2(mxa, mxb);
    mna = __hmin2(mna, mnb);
    nfa = __hadd2(nfa, nfb);
    mx = fmaxf(__low2float(mxa), __high2float(mxa));
    mn = fminf(__low2float(mna), __high2float(mna));
    nf = (__low2float(nfa) != 0.f || __high2float(nfa) != 0.f) ? 1.f : 0.f;
  } else {
    float mb = -INFINITY, nb = 0.f, lb = INFINITY;
    for (int j = 0; j < nfull; ++j) {
      float x[VE];
      Tr::values(mine[j], x);
      mx = fmaxf(mx, fmaxf(x[0], x[1]));
      mb = fmaxf(mb, fmaxf(x[2], x[3]));
      mn = fminf(mn, fminf(x[0], x[1]));
      lb = fminf(lb, fminf(x[2], x[3]));
      nf = fmaf(x[0], 0.f, fmaf(x[1], 0.f, nf));
      nb = fmaf(x[2], 0.f, fmaf(x[3], 0.f, nb));
    }
    mx = fmaxf(mx, mb);
    mn = fminf(mn, lb);
    nf += nb;
  }
  const int tail = thr_n - nfull * VE;
  if (tail) {
    float x[VE];
    Tr::values(mine[nfull], x);
#pragma unroll
    for (int i = 0; i < VE; ++i)
      if (i < tail) { mx = fmaxf(mx, x[i]); mn = fminf(mn, x[i]); nf = fmaf(x[i], 0.f, nf); }
  }
  nf_out = nf;
  mn_out = mn;
  return mx;
}

// ------------------------------------------------------------------------------------------------
// P4 main pass over one thread's vectors: one Philox4x32-10 word per kept token (x > xP, or x == xP and
// index <= It); returns the mask of vectors holding a kept token whose word is below bk. Vectors j < jfull
// lie at indices <= It, so only their values decide; in that range the pass draws four counters at a time
// (two bf16 vectors, four fp32 vectors) whenever every element of the group of vectors is kept.
// ------------------------------------------------------------------------------------------------
template <typename T>
static __device__ __noinline__ unsigned long long draw_scan(const uint4* mine, int thr_n, int64_t thr_e0, int jfull,
                                                           float xP, int32_t It, uint32_t g0, uint32_t rid,
                                                           uint32_t st_lo, uint32_t st_hi, uint32_t k0, uint32_t k1,
                                                           uint32_t bk) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  constexpr int G = VE / 4;            // counters per vector
  constexpr int U = 4 / G;             // vectors per step: four counters
  const PhiloxRow ph(PhiloxKey{k0, k1}, rid, st_lo, st_hi);
  const int nfull = thr_n / VE;
  const int nvec = (thr_n + VE - 1) / VE;
  unsigned long long flagged = 0ull;
  // one vector, any position: the groups of four tokens holding a kept token
  auto one = [&](int j) {
    float x[VE];
    Tr::values(mine[j], x);
    const int cnt = j < nfull ? VE : thr_n - nfull * VE;
    const int64_t e0 = thr_e0 + (int64_t)j * VE;
    uint32_t gmask = 0u;
#pragma unroll
    for (int i = 0; i < VE; ++i)
      if (i < cnt && (x[i] > xP || (x[i] == xP && e0 + i <= (int64_t)It))) gmask |= 1u << (i >> 2);
    if (!gmask) return;
    uint32_t bmin = 0xFFFFFFFFu;
#pragma unroll
    for (int g = 0; g < G; ++g)
      if ((gmask >> g) & 1u) bmin = min(bmin, min4_u32(ph(g0 + (uint32_t)(j * G + g))));
    if (bmin < bk) flagged |= 1ull << j;
  };
  int j = 0;
  for (; j + U <= jfull; j += U) {
    uint4 v[U];
    bool all = true;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      v[u] = mine[j + u];
      all = all && Tr::all_ge(v[u], xP);
    }
    if (all) {
      const uint32_t c0 = g0 + (uint32_t)(j * G);
      const uint4 w0 = ph(c0), w1 = ph(c0 + 1u), w2 = ph(c0 + 2u), w3 = ph(c0 + 3u);
      uint32_t m[4] = {min4_u32(w0), min4_u32(w1), min4_u32(w2), min4_u32(w3)};
#pragma unroll
      for (int u = 0; u < U; ++u) {
        uint32_t mu = m[u * G];
#pragma unroll
        for (int g = 1; g < G; ++g) mu = min(mu, m[u * G + g]);
        if (mu < bk) flagged |= 1ull << (j + u);
      }
    } else {
#pragma unroll 1
      for (int u = 0; u < U; ++u) one(j + u);
    }
  }
  for (; j < nvec; ++j) one(j);
  return flagged;
}

// The same over the vectors vis only (they hold every kept token).
template <typename T>
static __device__ __noinline__ unsigned long long draw_scan_in(const uint4* mine, int thr_n, int64_t thr_e0,
                                                           float xP, int32_t It, uint32_t g0, uint32_t rid,
                                                           uint32_t st_lo, uint32_t st_hi, uint32_t k0, uint32_t k1,
                                                           uint32_t bk, unsigned long long vis) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  constexpr int G = VE / 4;            // counters per vector
  const PhiloxRow ph(PhiloxKey{k0, k1}, rid, st_lo, st_hi);
  const int nfull = thr_n / VE;
  unsigned long long flagged = 0ull;
  // one vector, any position: the groups of four tokens holding a kept token
  auto one = [&](int j) {
    float x[VE];
    Tr::values(mine[j], x);
    const int cnt = j < nfull ? VE : thr_n - nfull * VE;
    const int64_t e0 = thr_e0 + (int64_t)j * VE;
    uint32_t gmask = 0u;
#pragma unroll
    for (int i = 0; i < VE; ++i)
      if (i < cnt && (x[i] > xP || (x[i] == xP && e0 + i <= (int64_t)It))) gmask |= 1u << (i >> 2);
    if (!gmask) return;
    uint32_t bmin = 0xFFFFFFFFu;
#pragma unroll
    for (int g = 0; g < G; ++g)
      if ((gmask >> g) & 1u) bmin = min(bmin, min4_u32(ph(g0 + (uint32_t)(j * G + g))));
    if (bmin < bk) flagged |= 1ull << j;
  };
  for (; vis; vis &= vis - 1ull) one(__ffsll((long long)vis) - 1);
  return flagged;
}

// ------------------------------------------------------------------------------------------------
// The kernel.
// ------------------------------------------------------------------------------------------------
// NDW data warps and one control warp per CTA; PER_SM CTAs resident per SM (the register budget).
template <typename T, int NDW, int PER_SM>
__global__ void __launch_bounds__((NDW + 1) * 32, PER_SM) sample_kernel(const Params p) {
  constexpr int kDataWarps = NDW;
  constexpr int kDataThreads = NDW * 32;
  constexpr int kSampleThreads = kDataThreads + 32;
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  constexpr int ES = Tr::ESIZE;
  extern __shared__ __align__(128) unsigned char dyn[];
  SampleSmem& sh = *reinterpret_cast<SampleSmem*>(dyn);
  unsigned char* slices = dyn + sample_slice_offset();   // p.nbuf buffers of one slice each
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int C = gridDim.x, crank = blockIdx.x;
  const int q = p.q;
  const int64_t G = gridDim.y;
  const int64_t first = blockIdx.y;
  const int64_t elems_cta = (int64_t)kDataThreads * q * VE;
  const int64_t cta_e0 = (int64_t)crank * elems_cta;
  const int64_t warp_bytes = (int64_t)32 * q * 16;

  if (t == 0) {
    for (int w = 0; w < kDataWarps; ++w) {
      mbar_init(&sh.lbar[0][w], 1);
      mbar_init(&sh.lbar[1][w], 1);
    }
    mbar_init(&sh.xbar[0], 1u);
    mbar_init(&sh.xbar[1], 1u);
    sh.acnt[0] = 0u;
    sh.acnt[1] = 0u;
    fence_mbar_init();
  }
  // every CTA's barriers are initialised before any peer can arrive on them
  cluster_barrier_shared();

  auto row_len = [&](int64_t r) -> int64_t {
    (void)r;
    return p.V;
  };

  if (warp < kDataWarps) {
    // =============================== data warps ===============================
    const int td = t;
    const int nbuf = p.nbuf > 1 ? 2 : 1;
    const int64_t slice_bytes = (int64_t)kDataThreads * q * 16;
    // After the slices, where the launch has room (p.vbytes): byte j * kDataThreads + td, the largest value bin of
    // vector j of thread td in the last value round; then four words per thread, word f * kDataThreads + td: vm
    // (f = 0, 1: the vectors with such a byte, those that matched that round) and km (f = 2, 3: the vectors
    // holding a key at or above the last REQ_MASS pivot). Kept in shared memory so they hold no registers
    // outside the radix requests.
    unsigned char* vbyte = p.vbytes ? slices + nbuf * slice_bytes : nullptr;
    uint32_t* vmw = p.vbytes ? reinterpret_cast<uint32_t*>(vbyte + ((int64_t)kDataThreads * q + 15) / 16 * 16) : nullptr;
    auto cta_count = [&](int64_t n) -> int64_t {
      const int64_t c = n - cta_e0;
      return c < 0 ? 0 : (c > elems_cta ? elems_cta : c);
    };
    // this warp's region of row r's slice into buffer b
    auto issue_warp = [&](int64_t r, int b) -> bool {
      const int64_t b16 = (cta_count(row_len(r)) * ES) & ~(int64_t)15;
      const int64_t lo = (int64_t)warp * warp_bytes;
      int64_t nb = b16 - lo;
      nb = nb < 0 ? 0 : (nb > warp_bytes ? warp_bytes : nb);
      mbar_arrive_expect_tx(&sh.lbar[b][warp], (uint32_t)nb);
      if (nb && !p.drop_loads) {
        bulk_copy_g2s(slices + b * slice_bytes + lo, p.x + ((int64_t)r * p.ld + cta_e0) * ES + lo, (uint32_t)nb,
                      &sh.lbar[b][warp]);
        return true;
      }
      return false;
    };
    // per buffer: completed phases, a copy armed and not yet waited for, a copy in flight
    int uses[2] = {0, 0};
    bool pending[2] = {false, false}, inflight[2] = {false, false};
    bool dead = false;
    if (p.tma) {
      for (int b = 0; b < nbuf; ++b) {
        if (first + b * G >= p.B) break;
        if (lane == 0) inflight[b] = issue_warp(first + b * G, b);
        pending[b] = true;
      }
    }

    for (int64_t k = 0;; ++k) {
      const int64_t row = first + k * G;
      if (row >= p.B) break;
      const int64_t n = row_len(row);
      const int64_t thr_e0 = cta_e0 + (int64_t)td * q * VE;
      int thr_n;
      {
        const int64_t r = n - thr_e0;
        thr_n = r < 0 ? 0 : (r > (int64_t)q * VE ? q * VE : (int)r);
      }
      const int nfull = thr_n / VE;
      const unsigned char* grow = p.x + ((int64_t)row * p.ld + cta_e0) * ES;
      const int buf = (int)(k % nbuf);
      unsigned char* slice = slices + buf * slice_bytes;
      const uint4* mine = reinterpret_cast<const uint4*>(slice) + (size_t)td * q;

      // ---- the slice ----
      bool timeout = dead;
      if (p.tma) {
        if (pending[buf] && !dead) {
          if (mbar_wait_bounded(&sh.lbar[buf][warp], (uint32_t)(uses[buf] & 1), p.wait_cycles)) {
            ++uses[buf];
            pending[buf] = false;
            inflight[buf] = false;
          } else {
            timeout = true;
          }
        }
        const int64_t cta_n = cta_count(n);
        const int64_t b16 = (cta_n * ES) & ~(int64_t)15;
        const int64_t tail_e0 = b16 / ES;
        if (!timeout && tail_e0 < cta_n && td == (int)(tail_e0 / ((int64_t)q * VE))) {
          for (int64_t e = tail_e0; e < cta_n; ++e) {
            if (ES == 4) reinterpret_cast<uint32_t*>(slice)[e] = reinterpret_cast<const uint32_t*>(grow)[e];
            else reinterpret_cast<uint16_t*>(slice)[e] = reinterpret_cast<const uint16_t*>(grow)[e];
          }
        }
      } else {
        for (int e = 0; e < thr_n; ++e) {
          const int64_t le = (int64_t)td * q * VE + e;
          if (ES == 4) reinterpret_cast<uint32_t*>(slice)[le] = reinterpret_cast<const uint32_t*>(grow)[le];
          else reinterpret_cast<uint16_t*>(slice)[le] = reinterpret_cast<const uint16_t*>(grow)[le];
        }
      }
      __syncwarp();   // the boundary search reads the chunks of the warp's other threads
      bool refilled = false;
      // after its last pass over this row the warp re-arms its region of this buffer with the row nbuf rows on
      auto refill = [&]() {
        if (refilled) return;
        refilled = true;
        const int64_t nr = row + nbuf * G;
        if (!p.tma || dead || nr >= p.B) return;
        __syncwarp();
        if (lane == 0) {
          fence_proxy_async_shared();
          inflight[buf] = issue_warp(nr, buf);
        }
        pending[buf] = true;
      };

      // ---- P1: maximum and non-finite check ----
      {
        float nf;
        float mn;
        float mx = max_pass<T>(mine, thr_n, nf, mn);
        const uint32_t flags = __reduce_or_sync(kFullMask, ((nf != 0.f) ? 1u : 0u) | (timeout ? 2u : 0u));
        mx = warp_max_f(mx);
        mn = -warp_max_f(-mn);
        if (lane == 0) sh.dp[warp][0] = make_uint4(__float_as_uint(mx), flags, __float_as_uint(mn), 0u);
        nb_arrive(SB_P1, kSampleThreads);
      }
      nb_sync(SB_CTL, kSampleThreads);
      const int status = sh.ctl.status;
      if (status == VSAMP_ERR_TIMEOUT) dead = true;
      if (status != VSAMP_OK) {
        refill();
        continue;
      }

      // ---- P2: fixed-point mass, maxima (with this thread's prefix inside the warp), min-p ----
      const float M = sh.ctl.M;
      uint32_t cm_thr, cm_pre;
      {
        const float c1 = sh.ctl.c1;
        const MassPart mp = sh.ctl.minp_on ? mass_pass<T, true>(mine, thr_n, M, c1, sh.ctl.kmin32)
                                           : mass_pass<T, false>(mine, thr_n, M, c1, 0u);
        uint32_t incl = mp.cm;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
          if (lane >= o) incl += y;
        }
        cm_thr = mp.cm;
        cm_pre = incl - mp.cm;
        const unsigned long long s = warp_sum_u64(mp.s);
        const uint32_t cm = __shfl_sync(kFullMask, incl, 31);
        unsigned long long mge = 0ull;
        uint32_t cge = 0u, minkey = 0xFFFFFFFFu, cmin = 0u;
        if (sh.ctl.minp_on) {
          mge = warp_sum_u64(mp.mge);
          cge = warp_sum_u32(mp.cge);
          minkey = warp_min_u32(mp.minkey);
          cmin = warp_sum_u32(mp.minkey == minkey ? mp.cmin : 0u);
        }
        if (lane == 0) {
          sh.dp[warp][0] = make_uint4((uint32_t)s, (uint32_t)(s >> 32), cm, cge);
          sh.dp[warp][1] = make_uint4((uint32_t)mge, (uint32_t)(mge >> 32), minkey, cmin);
        }
        nb_arrive(SB_P2, kSampleThreads);
      }

      // ---- requests of the control warp: radix histograms, tie counts ----
      uint32_t eq_thr = 0u, eq_pre = 0u;
      // vectors of this thread's chunk that held an element matching the previous round's prefix (bit j:
      // vector j; chunks of at most 64 vectors, longer ones visit every vector)
      const int nvec_thr = (thr_n + VE - 1) / VE;
      const bool masked = nvec_thr <= 64;
      uint32_t cand0 = 0u, cand1 = 0u;
      bool km_ok = false;            // this row's km words are valid
      // cand* reduced to the vectors whose largest bin in the last value round is at or above vsel
      auto by_bin = [&](uint32_t& m0, uint32_t& m1, int vsel) {
        uint32_t o0 = 0u, o1 = 0u;
        for (uint32_t bits = m0; bits; bits &= bits - 1u) {
          const int j = __ffs(bits) - 1;
          if ((int)vbyte[j * kDataThreads + td] >= vsel) o0 |= 1u << j;
        }
        for (uint32_t bits = m1; bits; bits &= bits - 1u) {
          const int j = __ffs(bits) - 1;
          if ((int)vbyte[(32 + j) * kDataThreads + td] >= vsel) o1 |= 1u << j;
        }
        m0 = o0;
        m1 = o1;
      };
      int req;
      for (;;) {
        nb_sync(SB_CTL, kSampleThreads);
        req = sh.ctl.req;
        if (req == REQ_DONE || req == REQ_ABORT) break;
        if (req == REQ_HIST) {
          const int shift = sh.ctl.shift, hp = sh.ctl.hpar;
          const bool hist_mass = sh.ctl.hist_mass != 0;
          const uint32_t prefix = sh.ctl.prefix;
          const uint32_t floor_rk = sh.ctl.floor_rk;
          const float c1 = sh.ctl.c1;
          const bool vround = sh.ctl.vround != 0;
          const ValueBins vb{sh.ctl.vxlo, sh.ctl.vsc};
          const uint32_t klo = sh.ctl.klo, khi = sh.ctl.khi;
          const int hi_shift = shift + 8;
          const uint32_t hmask = hi_shift >= 32 ? 0u : (0xFFFFFFFFu << hi_shift);
          uint32_t* hc = sh.hcnt[hp];
          unsigned long long* hm = sh.hm[hp];
          uint32_t run_bin = 0xFFFFFFFFu, run_cnt = 0;
          unsigned long long run_mass = 0;
          // the first key round after a value round: the smallest and largest matching key
          const bool track = !vround && sh.ctl.vsel >= 0;
          uint32_t kmn = 0xFFFFFFFFu, kmx = 0u;
          auto flush = [&]() {
            if (run_cnt) {
              atomicAdd(&hc[run_bin], run_cnt);
              if (hist_mass) atomicAdd(&hm[run_bin], run_mass);   // one 64-bit shared-memory add, no return
            }
          };
          // the vector's elements into the running bin; true if one matched
          auto visit = [&](int j) -> bool {
            float x[VE];
            Tr::values(mine[j], x);
            bool any = false;
            uint32_t vmax = 0u;
#pragma unroll
            for (int i = 0; i < VE; ++i) {
              if (j * VE + i >= thr_n) break;
              const uint32_t rk = Tr::rkey_of_value(x[i]);
              const bool match = vround ? rk >= floor_rk
                                        : ((rk & hmask) == (prefix & hmask) && rk >= floor_rk && rk >= klo && rk <= khi);
              if (match && track) {
                kmn = min(kmn, rk);
                kmx = max(kmx, rk);
              }
              if (match && !hist_mass) {
                // a count-only round: one atomic per element, no dependency from one element to the next
                any = true;
                const uint32_t bin = vround ? (uint32_t)value_bin(x[i], vb) : ((rk >> shift) & 255u);
                vmax = max(vmax, bin);
                atomicAdd(&hc[bin], 1u);
              } else if (match) {
                any = true;
                const uint32_t bin = vround ? (uint32_t)value_bin(x[i], vb) : ((rk >> shift) & 255u);
                vmax = max(vmax, bin);
                if (bin != run_bin) {
                  flush();
                  run_bin = bin;
                  run_cnt = 0;
                  run_mass = 0;
                }
                ++run_cnt;
                if (hist_mass) run_mass += mass_fx(ex2_approx((x[i] - M) * c1));
              }
            }
            if (vround && vbyte && j < 64) vbyte[j * kDataThreads + td] = (unsigned char)vmax;
            return any;
          };
          if (masked && sh.ctl.hfirst && vround && floor_rk == 0u && !hist_mass && !(sh.ctl.kfloor && km_ok)) {
            // the first round of a count search over the whole row
            value_round_full<T, kDataThreads>(mine, thr_n, vb, hc, vbyte, td);
            cand0 = nvec_thr >= 32 ? 0xFFFFFFFFu : ((1u << nvec_thr) - 1u);
            cand1 = nvec_thr >= 64 ? 0xFFFFFFFFu : (nvec_thr > 32 ? ((1u << (nvec_thr - 32)) - 1u) : 0u);
            if (vmw) {
              vmw[td] = cand0;
              vmw[kDataThreads + td] = cand1;
            }
          } else if (masked) {
            if (sh.ctl.hfirst) {   // the first round of a search visits every vector (with a floor: those above it)
              if (sh.ctl.kfloor && km_ok) {
                cand0 = vmw[2 * kDataThreads + td];
                cand1 = vmw[3 * kDataThreads + td];
              } else {
                cand0 = nvec_thr >= 32 ? 0xFFFFFFFFu : ((1u << nvec_thr) - 1u);
                cand1 = nvec_thr >= 64 ? 0xFFFFFFFFu : (nvec_thr > 32 ? ((1u << (nvec_thr - 32)) - 1u) : 0u);
              }
            } else if (sh.ctl.vsel >= 0 && vbyte) {
              // the first key round after a value round: the vectors holding a value in the selected bin or above
              by_bin(cand0, cand1, sh.ctl.vsel);
            }
            uint32_t next0 = 0u, next1 = 0u;
            if (!hist_mass) {
              // count-only rounds: two vectors per step (both loads issued before either is used), elements
              // predicated, one atomic per matching element
              auto count_vec = [&](const uint4 v, int j) -> bool {
                float x[VE];
                Tr::values(v, x);
                bool any = false;
                uint32_t vmax = 0u;
#pragma unroll
                for (int i = 0; i < VE; ++i) {
                  const uint32_t rk = Tr::rkey_of_value(x[i]);
                  const bool match = j * VE + i < thr_n &&
                      (vround ? rk >= floor_rk
                              : ((rk & hmask) == (prefix & hmask) && rk >= floor_rk && rk >= klo && rk <= khi));
                  if (match) {
                    any = true;
                    const uint32_t bin = vround ? (uint32_t)value_bin(x[i], vb) : ((rk >> shift) & 255u);
                    vmax = max(vmax, bin);
                    atomicAdd(&hc[bin], 1u);
                    if (track) {
                      kmn = min(kmn, rk);
                      kmx = max(kmx, rk);
                    }
                  }
                }
                if (vround && vbyte) vbyte[j * kDataThreads + td] = (unsigned char)vmax;
                return any;
              };
#pragma unroll
              for (int w = 0; w < 2; ++w) {
                uint32_t bits = w ? cand1 : cand0, hit = 0u;
                while (bits) {
                  const int b0 = __ffs(bits) - 1;
                  bits &= bits - 1u;
                  const int b1 = bits ? __ffs(bits) - 1 : b0;
                  const bool two = bits != 0u;
                  if (two) bits &= bits - 1u;
                  const uint4 v0 = mine[w * 32 + b0];
                  const uint4 v1 = mine[w * 32 + b1];
                  if (count_vec(v0, w * 32 + b0)) hit |= 1u << b0;
                  if (two && count_vec(v1, w * 32 + b1)) hit |= 1u << b1;
                }
                if (w) next1 = hit; else next0 = hit;
              }
            } else {
              for (uint32_t bits = cand0; bits; bits &= bits - 1u) {
                const int b = __ffs(bits) - 1;
                if (visit(b)) next0 |= 1u << b;
              }
              for (uint32_t bits = cand1; bits; bits &= bits - 1u) {
                const int b = __ffs(bits) - 1;
                if (visit(32 + b)) next1 |= 1u << b;
              }
            }
            cand0 = next0;
            cand1 = next1;
            if (vround && vmw) {
              vmw[td] = next0;
              vmw[kDataThreads + td] = next1;
            }
          } else {
            for (int j = 0; j * VE < thr_n; ++j) (void)visit(j);
          }
          flush();
          if (track) {
            kmn = __reduce_min_sync(kFullMask, kmn);
            kmx = __reduce_max_sync(kFullMask, kmx);
            if (lane == 0) sh.dp[warp][1] = make_uint4(kmn, kmx, 0u, 0u);
          }
        } else if (req == REQ_MASS) {   // fixed-point mass of the keys above a pivot, per warp
          const uint32_t rk0 = sh.ctl.prefix;
          const float c1 = sh.ctl.c1;
          unsigned long long sm = 0ull;
          uint32_t km0 = 0u, km1 = 0u;
          auto mass_vec = [&](int j) {
            float x[VE];
            Tr::values(mine[j], x);
            bool ge = false;
#pragma unroll
            for (int i = 0; i < VE; ++i) {
              const uint32_t rk = Tr::rkey_of_value(x[i]);
              if (j * VE + i < thr_n && rk > rk0) sm += mass_fx(ex2_approx((x[i] - M) * c1));
              ge = ge || (j * VE + i < thr_n && rk >= rk0);
            }
            if (ge && j < 64) {
              if (j < 32) km0 |= 1u << j;
              else km1 |= 1u << (j - 32);
            }
          };
          if (masked && vbyte && sh.ctl.vsel >= 0) {
            // keys at or above the pivot lie in its value bin or above: only the vectors reaching that bin
            uint32_t v0 = vmw[td], v1 = vmw[kDataThreads + td];
            by_bin(v0, v1, sh.ctl.vsel);
            for (uint32_t bits = v0; bits; bits &= bits - 1u) mass_vec(__ffs(bits) - 1);
            for (uint32_t bits = v1; bits; bits &= bits - 1u) mass_vec(32 + __ffs(bits) - 1);
          } else {
            for (int j = 0; j * VE < thr_n; ++j) mass_vec(j);
          }
          km_ok = masked && vmw;
          if (km_ok) {
            vmw[2 * kDataThreads + td] = km0;
            vmw[3 * kDataThreads + td] = km1;
          }
          sm = warp_sum_u64(sm);
          if (lane == 0) sh.dp[warp][0] = make_uint4((uint32_t)sm, (uint32_t)(sm >> 32), 0u, 0u);
        } else if (req == REQ_GATHER) {
          // the cluster's totals of this round's histograms, a bin per thread, into the other parity's arrays
          // (no peer reads those any more: every CTA has gathered the previous round before this exchange)
          const int hp = sh.ctl.hpar;
          const bool hm = sh.ctl.hist_mass != 0;
          for (int b = td; b < 256; b += kDataThreads) {
            uint32_t ct = 0u;
            unsigned long long mt = 0ull;
            for (int r0 = 0; r0 < C; r0 += 8) {
              uint32_t c[8];
              unsigned long long m[8];
#pragma unroll
              for (int r = 0; r < 8; ++r) {   // every load issued before any is used: one round trip
                c[r] = 0u;
                m[r] = 0ull;
                if (r0 + r < C) {
                  c[r] = dsmem_load_u32(dsmem_map(&sh.hcnt[hp][b], (uint32_t)(r0 + r)));
                  if (hm) m[r] = dsmem_load_u64(dsmem_map(&sh.hm[hp][b], (uint32_t)(r0 + r)));
                }
              }
#pragma unroll
              for (int r = 0; r < 8; ++r) {
                ct += c[r];
                mt += m[r];
              }
            }
            sh.hcnt[hp ^ 1][b] = ct;
            if (hm) sh.hm[hp ^ 1][b] = mt;
          }
        } else {   // REQ_COUNT: elements equal to xP, prefixed inside the warp
          const float xv = sh.ctl.xP;
          uint32_t c = 0;
          auto count_vec = [&](int j) {
            float x[VE];
            Tr::values(mine[j], x);
#pragma unroll
            for (int i = 0; i < VE; ++i) c += (j * VE + i < thr_n && x[i] == xv) ? 1u : 0u;
          };
          if (sh.ctl.kfloor && km_ok) {   // xP is at or above the top-k pivot: only the vectors holding such keys
            for (uint32_t bits = vmw[2 * kDataThreads + td]; bits; bits &= bits - 1u) count_vec(__ffs(bits) - 1);
            for (uint32_t bits = vmw[3 * kDataThreads + td]; bits; bits &= bits - 1u) count_vec(32 + __ffs(bits) - 1);
          } else {
            for (int j = 0; j * VE < thr_n; ++j) count_vec(j);
          }
          uint32_t incl = c;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
            if (lane >= o) incl += y;
          }
          eq_thr = c;
          eq_pre = incl - c;
          if (lane == 31) sh.dp[warp][0] = make_uint4(incl, 0u, 0u, 0u);
        }
        nb_arrive(SB_HIST, kSampleThreads);
      }
      if (req == REQ_ABORT) {
        if (sh.ctl.status == VSAMP_ERR_TIMEOUT) dead = true;
        refill();
        continue;
      }

      // ---- the cut's last kept element, per thread ----
      const int group = sh.ctl.group;
      float xP = group == GROUP_MAX ? M : sh.ctl.xP;
      int32_t It = kAllIndex;
      int32_t boundary = kNoIndex;
      if (group == GROUP_ALL) {
        xP = -INFINITY;
      } else if (group == GROUP_MAX || group == GROUP_PIVOT) {
        const unsigned long long need = sh.ctl.need;
        const unsigned long long start =
            (unsigned long long)sh.ctl.wstart[warp] + (group == GROUP_MAX ? cm_pre : eq_pre);
        const unsigned long long cnt = group == GROUP_MAX ? cm_thr : eq_thr;
        // warp-cooperative search of the boundary inside the chunk of the thread that holds it
        const bool holds = start < need && need <= start + cnt;
        const uint32_t bal = __ballot_sync(kFullMask, holds);
        if (bal) {
          const int src = __ffs(bal) - 1;
          uint32_t remaining = __shfl_sync(kFullMask, (uint32_t)(need - start), src);
          const int src_n = __shfl_sync(kFullMask, thr_n, src);
          const long long src_e0 = __shfl_sync(kFullMask, (long long)thr_e0, src);
          const uint4* src_vec = mine + (src - lane) * q;
          int32_t found = kNoIndex;
          for (int j0 = 0; j0 * VE < src_n; j0 += 32) {
            const int j = j0 + lane;
            const bool okv = j * VE < src_n;
            float x[VE];
            uint32_t c = 0;
            if (okv) {
              Tr::values(src_vec[j], x);
#pragma unroll
              for (int i = 0; i < VE; ++i) c += (j * VE + i < src_n && x[i] == xP) ? 1u : 0u;
            }
            uint32_t incl = c;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
              const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
              if (lane >= o) incl += y;
            }
            const uint32_t excl = incl - c;
            const bool here = okv && excl < remaining && remaining <= incl;
            int32_t idx = kNoIndex;
            if (here) {
              uint32_t seen = excl;
#pragma unroll
              for (int i = 0; i < VE; ++i)
                if (idx < 0 && j * VE + i < src_n && x[i] == xP && ++seen == remaining)
                  idx = (int32_t)(src_e0 + (long long)j * VE + i);
            }
            const uint32_t hb = __ballot_sync(kFullMask, here);
            if (hb) {
              found = __shfl_sync(kFullMask, idx, __ffs(hb) - 1);
              break;
            }
            remaining -= __shfl_sync(kFullMask, incl, 31);
          }
          if (lane == src) {
            boundary = found;
            It = found;
          } else {
            It = start >= need ? kNoIndex : kAllIndex;
          }
        } else {
          It = start >= need ? kNoIndex : kAllIndex;
        }
      }

      // ---- P4: Gumbel-max draw over the kept prefix ----
      if (sh.ctl.one_token) {
        // the first maximum: the boundary of a one-element cut
        int32_t b = boundary;
#pragma unroll
        for (int o = 16; o; o >>= 1) b = max(b, __shfl_xor_sync(kFullMask, b, o));
        if (lane == 0)
          sh.ap[warp] = make_uint4(__float_as_uint(-INFINITY), (uint32_t)(b >= 0 ? b : 0x7FFFFFFF), 0u, (uint32_t)b);
      } else {
        const bool all_cand = sh.ctl.all_cand != 0;
        const uint32_t bk = sh.ctl.bk;
        const uint32_t rid = sh.ctl.rid, st_lo = sh.ctl.st_lo, st_hi = sh.ctl.st_hi;
        const PhiloxKey key{sh.ctl.k0, sh.ctl.k1};
        int jfull = 0;
        {
          const int64_t lim = (int64_t)It - thr_e0 - (VE - 1);
          if (lim >= 0) jfull = (int)(lim / VE + 1 < (int64_t)nfull ? lim / VE + 1 : (int64_t)nfull);
        }
        const uint32_t g0 = (uint32_t)(thr_e0 >> 2);
        // after a top-k search every kept token lies in a vector holding a key at or above its pivot
        const unsigned long long vis = (sh.ctl.p4km && km_ok)
            ? (((unsigned long long)vmw[3 * kDataThreads + td] << 32) | vmw[2 * kDataThreads + td]) : ~0ull;
        unsigned long long flagged =
            all_cand ? kept_vectors_in<T>(mine, thr_n, thr_e0, xP, It, vis)
            : vis != ~0ull
                ? draw_scan_in<T>(mine, thr_n, thr_e0, xP, It, g0, rid, st_lo, st_hi, key.k0, key.k1, bk, vis)
                : draw_scan<T>(mine, thr_n, thr_e0, jfull, xP, It, g0, rid, st_lo, st_hi, key.k0, key.k1, bk);
        // flagged vectors: the kept tokens whose word passes the bound get the exact perturbed score
        float bscore = -INFINITY, bs = 0.f;
        int32_t bidx = 0x7FFFFFFF;
        if (flagged) {
          const float invT = sh.ctl.invT, c1 = sh.ctl.c1, kappa = sh.ctl.kappa;
          while (flagged) {
            const int j = __ffsll((long long)flagged) - 1;
            flagged &= flagged - 1ull;
            float x[VE];
            Tr::values(mine[j], x);
            const int cnt = j < nfull ? VE : thr_n - nfull * VE;
            const int64_t e0 = thr_e0 + (int64_t)j * VE;
            uint32_t b[VE];
#pragma unroll
            for (int g = 0; g < VE / 4; ++g) {
              const uint4 w4 = philox4x32_10(make_uint4(g0 + (uint32_t)(j * (VE / 4) + g), rid, st_lo, st_hi), key);
              b[4 * g + 0] = w4.x; b[4 * g + 1] = w4.y; b[4 * g + 2] = w4.z; b[4 * g + 3] = w4.w;
            }
#pragma unroll
            for (int i = 0; i < VE; ++i) {
              if (!(i < cnt && (x[i] > xP || (x[i] == xP && e0 + i <= (int64_t)It)))) continue;
              if (!all_cand && b[i] >= bk) continue;
              const float d = x[i] - M;
              const float s = d * invT;
              if (!all_cand) {
                const float w = ex2_approx(d * c1);
                const float u = fmaf((float)b[i], kTwoM32, kTwoM33);
                if (!(u < w * kappa * 1.00001f)) continue;
              }
              const float score = gumbel_score(s, b[i]);
              const int32_t idx = (int32_t)(e0 + i);
              if (argmax_better(score, idx, bscore, bidx)) { bscore = score; bidx = idx; bs = s; }
            }
          }
        }
        const ArgMax best = warp_argmax(ArgMax{bscore, bidx, bs});
        int32_t wcut = boundary;
#pragma unroll
        for (int o = 16; o; o >>= 1) wcut = max(wcut, __shfl_xor_sync(kFullMask, wcut, o));
        if (lane == 0)
          sh.ap[warp] = make_uint4(__float_as_uint(best.score), (uint32_t)best.idx, __float_as_uint(best.s), (uint32_t)wcut);
      }
      nb_arrive(SB_P4, kSampleThreads);
      refill();
    }
    // a bulk copy of this warp that may still be landing in shared memory (after a timed-out load)
    for (int b = 0; b < nbuf; ++b)
      if (p.tma && inflight[b]) (void)mbar_wait_bounded(&sh.lbar[b][warp], (uint32_t)(uses[b] & 1), 4000000000LL);
  } else {
    // =============================== control warp ===============================
    ClusterXchg X;
    int hround = 0;          // radix rounds so far (histogram buffer parity)
    bool dead = false;       // an exchange timed out: later rows are reported as timed out
    const unsigned long long one = 1ull << kMassShift;
    for (int64_t k = 0;; ++k) {
      const int64_t row = first + k * G;
      if (row >= p.B) break;
      const int64_t n = row_len(row);
      float temp = 1.f, topp = 1.f, minp = 0.f;
      int32_t topk = 0;
      if (p.temperature) temp = p.temperature[row];
      if (p.top_k) topk = p.top_k[row];
      if (p.top_p) topp = p.top_p[row];
      if (p.min_p) minp = p.min_p[row];
      uint64_t sd = 0ull, st = 0ull;
      uint32_t rid = (uint32_t)row;
      if (p.seed) sd = p.seed[row];
      if (p.step) st = p.step[row];
      if (p.row_id) rid = p.row_id[row];
      int passes = 1, rounds = 0, path = p.tma ? 0 : PATH_NOTMA;

      // ---- P1 partials -> cluster maximum and minimum ----
      nb_sync(SB_P1, kSampleThreads);
      float M, Mmin;
      uint32_t flags;
      {
        float m = -INFINITY, m2 = INFINITY;
        uint32_t fl = 0u;
        if (lane < kDataWarps) {
          const uint4 v = sh.dp[lane][0];
          m = __uint_as_float(v.x);
          fl = v.y;
          m2 = __uint_as_float(v.z);
        }
        m = warp_max_f(m);
        m2 = -warp_max_f(-m2);
        fl = __reduce_or_sync(kFullMask, fl);
        if (!dead) {
          if (!X.run(sh, C, crank, make_uint4(__float_as_uint(m), fl, __float_as_uint(m2), 0u),
                     make_uint4(0u, 0u, 0u, 0u), p.wait_cycles))
            dead = true;
        }
        m = -INFINITY;
        m2 = INFINITY;
        fl = dead ? 2u : 0u;
        if (!dead && lane < C) {
          const uint4 v = sh.xm[X.par() ^ 1][lane][0];
          m = __uint_as_float(v.x);
          fl |= v.y;
          m2 = __uint_as_float(v.z);
        }
        M = warp_max_f(m);
        Mmin = -warp_max_f(-m2);
        flags = __reduce_or_sync(kFullMask, fl);
        if (flags & 2u) dead = true;
      }
      int status = VSAMP_OK;
      if (flags & 2u) status = VSAMP_ERR_TIMEOUT;
      else if (flags & 1u) status = VSAMP_ERR_NONFINITE;
      else if (isnan(temp) || isinf(temp) || isnan(topp) || !(topp > 0.f) || isnan(minp) || minp > 1.f)
        status = VSAMP_ERR_INVALID_ARG;
      const bool greedy = !(temp > 0.f);
      const float Teff = greedy ? 1.f : temp;
      const float invT = 1.f / Teff;
      const float c1 = kLog2e * invT;
      bool minp_on = !greedy && minp > 0.f;
      uint32_t kmin32 = 0u;
      if (minp_on && status == VSAMP_OK) {
        // min-p keeps w >= minp <=> x >= x* = M + T ln(minp), formed as an unevaluated sum; the threshold
        // is the smallest fp32 value >= x*
        const float L = logf(minp);
        const float ph = Teff * L, pl = fmaf(Teff, L, -ph);
        const float sh_ = M + ph;
        const float bb = sh_ - M;
        const float sl = (M - (sh_ - bb)) + (ph - bb);
        const float lo = sl + pl;
        const float xf = lo > 0.f ? nextafterf(sh_, INFINITY) : sh_;
        kmin32 = key_f32_bits(__float_as_uint(xf));
        // a threshold at or below the row's minimum keeps every token: the filter is off
        if (kmin32 <= key_f32_bits(__float_as_uint(Mmin))) minp_on = false;
      }
      if (lane == 0) {
        sh.ctl.status = status;
        sh.ctl.M = M;
        sh.ctl.c1 = c1;
        sh.ctl.invT = invT;
        sh.ctl.minp_on = minp_on ? 1 : 0;
        sh.ctl.kmin32 = kmin32;
      }
      __syncwarp();
      nb_arrive(SB_CTL, kSampleThreads);

      auto write_error = [&](int st_code) {
        if (crank == 0 && lane == 0) {
          p.token[row] = -1;
          if (p.logprob) p.logprob[row] = __int_as_float(0x7FC00000);
          if (p.row_status) p.row_status[row] = st_code;
          if (p.stats) {
            p.stats[row * 4 + 0] = passes;
            p.stats[row * 4 + 1] = rounds;
            p.stats[row * 4 + 2] = 0;
            p.stats[row * 4 + 3] = p.tma ? 0 : PATH_NOTMA;
          }
        }
      };
      if (status != VSAMP_OK) {
        write_error(status);
        continue;
      }

      // ---- P2 partials -> cluster mass, maxima, min-p statistics ----
      passes = 2;
      nb_sync(SB_P2, kSampleThreads);
      unsigned long long Sfx, mass_ge = 0ull;
      uint32_t cM, cm_before = 0u, cnt_ge = 0u, minkey_ge = 0xFFFFFFFFu, cnt_minkey = 0u;
      uint32_t wpre_max = 0u;   // lane w < kDataWarps: maxima of the CTA's warps before w
      bool xok = true;
      {
        unsigned long long a = 0ull, b = 0ull;
        uint32_t c = 0u, d = 0u, mk = 0xFFFFFFFFu, cc = 0u;
        if (lane < kDataWarps) {
          const uint4 v0 = sh.dp[lane][0], v1 = sh.dp[lane][1];
          a = u64_of(v0.x, v0.y);
          c = v0.z;
          d = v0.w;
          b = u64_of(v1.x, v1.y);
          mk = v1.z;
          cc = v1.w;
        }
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
          if (lane >= o) incl += y;
        }
        wpre_max = incl - c;
        a = warp_sum_u64(a);
        c = __shfl_sync(kFullMask, incl, 31);
        if (minp_on) {
          b = warp_sum_u64(b);
          d = warp_sum_u32(d);
          const uint32_t gmk = warp_min_u32(mk);
          cc = warp_sum_u32(mk == gmk ? cc : 0u);
          mk = gmk;
        }
        xok = X.run(sh, C, crank, make_uint4((uint32_t)a, (uint32_t)(a >> 32), c, d),
                    make_uint4((uint32_t)b, (uint32_t)(b >> 32), mk, cc), p.wait_cycles);
        a = 0ull; b = 0ull; c = 0u; d = 0u; mk = 0xFFFFFFFFu; cc = 0u;
        if (lane < C) {
          const uint4 v0 = sh.xm[X.par() ^ 1][lane][0], v1 = sh.xm[X.par() ^ 1][lane][1];
          a = u64_of(v0.x, v0.y);
          c = v0.z;
          d = v0.w;
          b = u64_of(v1.x, v1.y);
          mk = v1.z;
          cc = v1.w;
        }
        uint32_t ci = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(kFullMask, ci, o);
          if (lane >= o) ci += y;
        }
        cm_before = __shfl_sync(kFullMask, ci - c, crank);
        Sfx = warp_sum_u64(a);
        cM = __shfl_sync(kFullMask, ci, 31);
        if (minp_on) {
          mass_ge = warp_sum_u64(b);
          cnt_ge = warp_sum_u32(d);
          minkey_ge = warp_min_u32(mk);
          cnt_minkey = warp_sum_u32(mk == minkey_ge ? cc : 0u);
        }
      }
      auto abort_row = [&](int st_code) {
        if (lane == 0) {
          sh.ctl.status = st_code;
          sh.ctl.req = REQ_ABORT;
        }
        __syncwarp();
        nb_arrive(SB_CTL, kSampleThreads);
        write_error(st_code);
      };
      if (!xok) {
        dead = true;
        abort_row(VSAMP_ERR_TIMEOUT);
        continue;
      }

      // ---- plan: the shortest prefix over top-k, top-p and min-p ----
      const float logS = logf(u64_to_float(Sfx) * 9.094947017729282379e-13f);   // 2^-40
      const uint32_t rkM = Tr::rkey_of_value(M);
      int plan_status = VSAMP_OK;
      int ck_mode = 0, cp_mode = 0;
      float goal_p = -1.f;
      unsigned long long cp_goal = 0ull;
      Cut ck{}, cp{}, fin{};
      // one radix search, driven through the data warps; false on an exchange timeout
      // floor_rk: keys below it are left out of the histograms (only where the goal is reached within the keys
      // at or above it, so the group found and its counts do not change)
      auto radix = [&](bool mass_mode, unsigned long long goal, float gp, bool want_mass, uint32_t floor_rk,
                       RadixOut& out) -> bool {
        out = RadixOut{};
        out.ok = 1;
        out.vsel = -1;
        int vsel_next = -1;   // the next request is the first key round after the value round
        int vsel_cur = -1;    // this request is
        uint32_t prefix = 0;
        unsigned long long cnt_above = 0, mass_above = 0;
        const bool hist_mass = want_mass || mass_mode;
        // the first round bins values linearly over the candidates' range when it is finite (ValueBins)
        const float xlo = floor_rk ? fmaxf(Mmin, Tr::value_of_rkey(floor_rk)) : Mmin;
        const ValueBins vb = make_value_bins(xlo, M);
        bool vround = vb.sc > 0.f, first = true;
        uint32_t klo = 0u, khi = 0xFFFFFFFFu;
        int shift = vround ? 0 : Tr::KB - 8;
        for (;;) {
          const int hp = hround & 1;
          ++hround;
          for (int b = lane; b < 256; b += 32) {
            sh.hcnt[hp][b] = 0u;
            sh.hm[hp][b] = 0ull;
          }
          if (lane == 0) {
            sh.ctl.req = REQ_HIST;
            sh.ctl.shift = shift;
            sh.ctl.hpar = hp;
            sh.ctl.hist_mass = hist_mass ? 1 : 0;
            sh.ctl.prefix = prefix;
            sh.ctl.floor_rk = floor_rk;
            sh.ctl.hfirst = first ? 1 : 0;
            sh.ctl.kfloor = floor_rk != 0u ? 1 : 0;
            sh.ctl.vround = vround ? 1 : 0;
            sh.ctl.vxlo = vb.xlo;
            sh.ctl.vsc = vb.sc;
            sh.ctl.klo = klo;
            sh.ctl.khi = khi;
            sh.ctl.vsel = vsel_next;
          }
          vsel_cur = vsel_next;
          vsel_next = -1;
          __syncwarp();
          nb_arrive(SB_CTL, kSampleThreads);
          nb_sync(SB_HIST, kSampleThreads);
          ++passes;
          ++rounds;
          // the first key round after a value round: the CTA's smallest and largest matching key travel with
          // the exchange; when the cluster's are equal (a bin holding one distinct value) the search ends there
          const bool track = vsel_cur >= 0;
          uint32_t kmn = 0xFFFFFFFFu, kmx = 0u;
          if (track && lane < kDataWarps) {
            kmn = sh.dp[lane][1].x;
            kmx = sh.dp[lane][1].y;
          }
          if (track) {
            kmn = __reduce_min_sync(kFullMask, kmn);
            kmx = __reduce_max_sync(kFullMask, kmx);
          }
          // every CTA's histogram is complete once every CTA has passed this exchange
          if (!X.run(sh, C, crank, make_uint4(kmn, kmx, 0u, 0u), make_uint4(0u, 0u, 0u, 0u), p.wait_cycles)) return false;
          if (track) {
            uint32_t a = 0xFFFFFFFFu, z = 0u;
            if (lane < C) {
              const uint4 m = sh.xm[X.par() ^ 1][lane][0];
              a = m.x;
              z = m.y;
            }
            kmn = __reduce_min_sync(kFullMask, a);
            kmx = __reduce_max_sync(kFullMask, z);
          }
          int sp = hp;   // the arrays holding the cluster's totals
          if (C > 1) {   // the data warps sum the peers' histograms, a bin per thread, into the other parity
            if (lane == 0) sh.ctl.req = REQ_GATHER;
            __syncwarp();
            nb_arrive(SB_CTL, kSampleThreads);
            nb_sync(SB_HIST, kSampleThreads);
            sp = hp ^ 1;
          }
          // lane l: bins 255 - 8l .. 248 - 8l (32-byte aligned: two 16-byte loads per array)
          uint32_t bc[8];
          unsigned long long bm[8];
          {
            const int b0 = 248 - 8 * lane;
            const uint4 c0 = *reinterpret_cast<const uint4*>(&sh.hcnt[sp][b0]);
            const uint4 c1 = *reinterpret_cast<const uint4*>(&sh.hcnt[sp][b0 + 4]);
            ulonglong2 m01 = make_ulonglong2(0ull, 0ull), m23 = m01, m45 = m01, m67 = m01;
            if (hist_mass) {
              m01 = *reinterpret_cast<const ulonglong2*>(&sh.hm[sp][b0]);
              m23 = *reinterpret_cast<const ulonglong2*>(&sh.hm[sp][b0 + 2]);
              m45 = *reinterpret_cast<const ulonglong2*>(&sh.hm[sp][b0 + 4]);
              m67 = *reinterpret_cast<const ulonglong2*>(&sh.hm[sp][b0 + 6]);
            }
            // bc[i] / bm[i] hold bin 255 - 8l - i = b0 + 7 - i
            const uint32_t cc[8] = {c1.w, c1.z, c1.y, c1.x, c0.w, c0.z, c0.y, c0.x};
            const unsigned long long mm[8] = {m67.y, m67.x, m45.y, m45.x, m23.y, m23.x, m01.y, m01.x};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              bc[i] = cc[i];
              bm[i] = mm[i];
            }
          }
          if (mass_mode && gp >= 0.f && first) {
            unsigned long long tot = 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) tot += bm[i];
            tot = warp_sum_u64(tot);
            goal = ceil_mul_frac(gp, tot);
          }
          uint32_t lc = 0;
          unsigned long long lm = 0;
#pragma unroll
          for (int i = 0; i < 8; ++i) { lc += bc[i]; lm += bm[i]; }
          uint32_t ic = lc;
          unsigned long long im = lm;
#pragma unroll
          for (int o = 1; o < 32; o <<= 1) {
            const uint32_t yc = __shfl_up_sync(kFullMask, ic, o);
            const unsigned long long ym = __shfl_up_sync(kFullMask, im, o);
            if (lane >= o) { ic += yc; im += ym; }
          }
          const unsigned long long ec = ic - lc, em = im - lm;   // bins above this lane's
          const bool mine_has = mass_mode ? (em < goal && goal <= im) : (ec < goal && goal <= (unsigned long long)ic);
          const uint32_t ballot = __ballot_sync(kFullMask, mine_has);
          if (ballot == 0) {   // cannot happen with consistent histograms; reported as an error
            out.ok = 0;
            return true;
          }
          const int src = __ffs(ballot) - 1;
          uint32_t sel = 0xFFFFFFFFu;
          unsigned long long ac = ec, am = em, ceq = 0, meq = 0;
          if (lane == src) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const unsigned long long c = bc[i], m = bm[i];
              const bool hit = mass_mode ? (am < goal && goal <= am + m) : (ac < goal && goal <= ac + c);
              if (hit && sel == 0xFFFFFFFFu) { sel = (uint32_t)(255 - 8 * lane - i); ceq = c; meq = m; }
              if (sel == 0xFFFFFFFFu) { ac += c; am += m; }
            }
          }
          sel = __shfl_sync(kFullMask, sel, src);
          ac = __shfl_sync(kFullMask, ac, src);
          am = __shfl_sync(kFullMask, am, src);
          ceq = __shfl_sync(kFullMask, ceq, src);
          meq = __shfl_sync(kFullMask, meq, src);
          out.cnt_eq = ceq;
          out.mass_eq = meq;
          cnt_above += ac;
          mass_above += am;
          if (mass_mode) goal -= am; else goal -= ac;
          first = false;
          if (vround) {
            // the selected value bin's key range, then key rounds inside it
            const KeyRange kr = key_range_of_bin<Tr>((int)sel, Tr::rkey_of_value(xlo), Tr::rkey_of_value(M), vb);
            vround = false;
            klo = kr.klo;
            khi = kr.khi;
            prefix = kr.prefix;
            out.vsel = (int)sel;
            vsel_next = (int)sel;
            if (kr.shift < 0) break;   // one key: the group
            shift = kr.shift;
            continue;
          }
          if (track && kmn == kmx) {   // every matching element holds the same key: the group
            prefix = kmn;
            break;
          }
          prefix |= sel << shift;
          if (shift == 0) break;
          shift -= 8;
        }
        out.rk = prefix;
        out.cnt_above = cnt_above;
        out.mass_above = mass_above;
        out.goal = goal;
        return true;
      };

      if (greedy) {
        fin = Cut{rkM, 0, 1, cM, one, 0};
        path |= PATH_MAXGROUP;
      } else {
        const bool topk_on = topk > 0 && (int64_t)topk < n;
        const bool topp_on = topp < 1.f;
        const unsigned long long keff = topk_on ? (unsigned long long)topk : (unsigned long long)n;
        if (topk_on) {
          if (keff <= cM) {
            ck = Cut{rkM, 0, keff, cM, keff * one, 0};
            ck_mode = 1;
          } else {
            ck = Cut{0, 0, keff, 0, 0, 0};
            ck_mode = 2;
          }
        }
        if (topp_on) {
          if (ck_mode != 2) {
            const unsigned long long Sk = topk_on ? ck.mass : Sfx;
            const unsigned long long target = ceil_mul_frac(topp, Sk);
            if (target <= cM * one) {
              unsigned long long need = (target + one - 1) >> kMassShift;
              need = need < 1 ? 1 : need;
              cp = Cut{rkM, 0, need, cM, need * one, 0};
              cp_mode = 1;
            } else {
              cp_mode = 2;
              if (topk_on) cp_goal = target;
              else goal_p = topp;
            }
          } else if (ceil_mul_frac(topp, Sfx) <= one) {
            cp = Cut{rkM, 0, 1, cM, one, 0};
            cp_mode = 1;
          } else {
            cp_mode = 2;
          }
        }
        // top-p keeping the first maximum alone is the shortest cut: no radix search for top-k
        if (cp_mode == 1 && cp.kept() == 1 && ck_mode == 2) ck_mode = 0;
        if (ck_mode == 1 || cp_mode == 1) path |= PATH_MAXGROUP;
        if (minp_on) {
          const uint32_t rkm = (Tr::KB == 32) ? minkey_ge : (minkey_ge >> 16);
          fin = Cut{rkm, (unsigned long long)(cnt_ge - cnt_minkey), cnt_minkey, cnt_minkey, mass_ge, 1};
        } else {
          fin = Cut{rkM, 0, (unsigned long long)n, 0, Sfx, 1};
        }
        bool rok = true;
        if (ck_mode == 2) {
          // a count search, then the kept mass (the top-p goal and the prune bound of the draw use it) in one
          // pass over the keys above the pivot
          RadixOut r;
          rok = radix(false, ck.need, -1.f, false, 0u, r);
          unsigned long long above = 0ull;
          if (rok && r.ok) {
            if (lane == 0) {
              sh.ctl.req = REQ_MASS;
              sh.ctl.prefix = r.rk;
              sh.ctl.vsel = r.vsel;
            }
            __syncwarp();
            nb_arrive(SB_CTL, kSampleThreads);
            nb_sync(SB_HIST, kSampleThreads);
            ++passes;
            unsigned long long w = 0ull;
            if (lane < kDataWarps) w = ((unsigned long long)sh.dp[lane][0].y << 32) | sh.dp[lane][0].x;
            w = warp_sum_u64(w);
            rok = X.run(sh, C, crank, make_uint4((uint32_t)w, (uint32_t)(w >> 32), 0u, 0u),
                        make_uint4(0u, 0u, 0u, 0u), p.wait_cycles);
            if (rok) {
              unsigned long long a = 0ull;
              if (lane < C) {
                const uint4 m = sh.xm[X.par() ^ 1][lane][0];
                a = ((unsigned long long)m.y << 32) | m.x;
              }
              above = warp_sum_u64(a);
            }
          }
          if (rok) {
            if (!r.ok) plan_status = VSAMP_ERR_INVALID_ARG;
            const unsigned long long need = ck.need - r.cnt_above;
            const unsigned long long wP = mass_fx(ex2_approx((Tr::value_of_rkey(r.rk) - M) * c1));
            ck = Cut{r.rk, r.cnt_above, need, r.cnt_eq, above + need * wP, 0};
            path |= PATH_RADIX_K;
            if (cp_mode == 2) cp_goal = ceil_mul_frac(topp, ck.mass);
          }
        }
        if (rok && cp_mode == 2 && plan_status == VSAMP_OK) {
          RadixOut r;
          // after a top-k cut the goal lies within the keys at or above its pivot
          rok = radix(true, cp_goal, goal_p, true, ck_mode == 2 ? ck.rk : 0u, r);
          if (rok) {
            if (!r.ok) plan_status = VSAMP_ERR_INVALID_ARG;
            const unsigned long long wP = mass_fx(ex2_approx((Tr::value_of_rkey(r.rk) - M) * c1));
            unsigned long long need = wP ? (r.goal + wP - 1) / wP : 1;
            need = need < 1 ? 1 : (need > r.cnt_eq ? r.cnt_eq : need);
            cp = Cut{r.rk, r.cnt_above, need, r.cnt_eq, r.mass_above + need * wP, 0};
            path |= PATH_RADIX_P;
          }
        }
        if (!rok) {
          dead = true;
          abort_row(VSAMP_ERR_TIMEOUT);
          continue;
        }
        Cut best = fin;
        if (ck_mode && ck.kept() < best.kept()) best = ck;
        if (cp_mode && cp.kept() < best.kept()) best = cp;
        if (minp_on && best.whole) path |= PATH_MINP;
        fin = best;
      }
      if (plan_status != VSAMP_OK) {
        abort_row(plan_status);
        continue;
      }

      // ---- the cut handed to the data warps ----
      const unsigned long long kept = fin.kept();
      const bool one_token = greedy || kept == 1;
      const bool need_boundary = !fin.whole || one_token;
      int group;
      unsigned long long need = fin.need;
      uint32_t wstart = 0u;   // lane w < kDataWarps
      float xP = Tr::value_of_rkey(fin.rk);
      if (!need_boundary) {
        group = (fin.above == 0 && fin.cnt_eq == 0) ? GROUP_ALL : GROUP_WHOLE;
        if (group == GROUP_ALL) xP = -INFINITY;
      } else if (fin.rk == rkM) {
        group = GROUP_MAX;
        if (fin.whole) need = cM;
        wstart = cm_before + wpre_max;
      } else {
        group = GROUP_PIVOT;
        if (lane == 0) {
          sh.ctl.req = REQ_COUNT;
          sh.ctl.xP = xP;
          sh.ctl.kfloor = ck_mode == 2 ? 1 : 0;
        }
        __syncwarp();
        nb_arrive(SB_CTL, kSampleThreads);
        nb_sync(SB_HIST, kSampleThreads);
        ++passes;
        uint32_t c = lane < kDataWarps ? sh.dp[lane][0].x : 0u;
        uint32_t incl = c;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
          if (lane >= o) incl += y;
        }
        const uint32_t wpre = incl - c;
        const uint32_t ctot = __shfl_sync(kFullMask, incl, 31);
        if (!X.run(sh, C, crank, make_uint4(ctot, 0u, 0u, 0u), make_uint4(0u, 0u, 0u, 0u), p.wait_cycles)) {
          dead = true;
          abort_row(VSAMP_ERR_TIMEOUT);
          continue;
        }
        const uint32_t v = lane < C ? sh.xm[X.par() ^ 1][lane][0].x : 0u;
        uint32_t vi = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t y = __shfl_up_sync(kFullMask, vi, o);
          if (lane >= o) vi += y;
        }
        const uint32_t cpre = __shfl_sync(kFullMask, vi - v, crank);
        const uint32_t total = __shfl_sync(kFullMask, vi, 31);
        if (fin.whole) need = total;
        wstart = cpre + wpre;
      }

      // ---- the draw's prune bound: a token can beat B0 = ln(S_kept) - 3 only if u < w * kappa ----
      float kappa = 0.f, B0 = 0.f;
      bool all_cand = false;
      uint32_t bk = 0u;
      if (!one_token) {
        const float skept = fmaxf(u64_to_float(fin.mass) * 9.094947017729282379e-13f, 1.f);
        kappa = 20.085536923187668f / skept;
        all_cand = kappa >= 0.99f;
        bk = all_cand ? 0xFFFFFFFFu : __float2uint_ru(kappa * 1.00001f * 4294967296.0f);
        B0 = -logf(kappa);
        ++passes;
      }
      if (lane < kDataWarps) sh.ctl.wstart[lane] = wstart;
      if (lane == 0) {
        sh.ctl.req = REQ_DONE;
        sh.ctl.p4km = ck_mode == 2 ? 1 : 0;   // the cut lies at or above the top-k pivot
        sh.ctl.group = group;
        sh.ctl.xP = xP;
        sh.ctl.need = need;
        sh.ctl.one_token = one_token ? 1 : 0;
        sh.ctl.all_cand = all_cand ? 1 : 0;
        sh.ctl.bk = bk;
        sh.ctl.kappa = kappa;
        sh.ctl.rid = rid;
        sh.ctl.st_lo = (uint32_t)st;
        sh.ctl.st_hi = (uint32_t)(st >> 32);
        sh.ctl.k0 = (uint32_t)sd;
        sh.ctl.k1 = (uint32_t)(sd >> 32);
      }
      __syncwarp();
      nb_arrive(SB_CTL, kSampleThreads);

      // ---- P4 partials -> the cluster arg-max (lock-free: the last CTA to publish writes the outputs) ----
      nb_sync(SB_P4, kSampleThreads);
      ArgMax c2{-INFINITY, 0x7FFFFFFF, 0.f};
      int32_t ccut = -1;
      if (lane < kDataWarps) {
        const uint4 v = sh.ap[lane];
        c2 = ArgMax{__uint_as_float(v.x), (int32_t)v.y, __uint_as_float(v.z)};
        ccut = (int32_t)v.w;
      }
      c2 = warp_argmax(c2);
#pragma unroll
      for (int o = 16; o; o >>= 1) ccut = max(ccut, __shfl_xor_sync(kFullMask, ccut, o));
      const int par = (int)(k & 1);
      uint32_t old = 0u;
      if (C > 1 && lane == 0) {
        dsmem_store_v4(dsmem_map(&sh.aslot[par][crank], 0), __float_as_uint(c2.score), (uint32_t)c2.idx,
                       __float_as_uint(c2.s), (uint32_t)ccut);
        old = dsmem_atomic_add_acq_rel(dsmem_map(&sh.acnt[par], 0), 1u);
      }
      old = __shfl_sync(kFullMask, old, 0);
      if (C > 1 && old != (uint32_t)(C - 1)) continue;   // another CTA writes the outputs
      __syncwarp();
      ArgMax g = c2;
      int32_t cut = ccut;
      if (C > 1) {
        g = ArgMax{-INFINITY, 0x7FFFFFFF, 0.f};
        cut = -1;
        if (lane < C) {
          const uint4 v = dsmem_load_v4(dsmem_map(&sh.aslot[par][lane], 0));
          g = ArgMax{__uint_as_float(v.x), (int32_t)v.y, __uint_as_float(v.z)};
          cut = (int32_t)v.w;
        }
        g = warp_argmax(g);
#pragma unroll
        for (int o = 16; o; o >>= 1) cut = max(cut, __shfl_xor_sync(kFullMask, cut, o));
        if (lane == 0) dsmem_store_u32(dsmem_map(&sh.acnt[par], 0), 0u);
      }
      int32_t out_token;
      float out_s;
      if (one_token) {
        out_token = g.idx;
        out_s = 0.f;   // a maximum: (x - M) / T = 0
      } else if (all_cand || g.score > B0 + 1e-4f * fmaxf(1.f, fabsf(B0))) {
        out_token = g.idx;
        out_s = g.s;
      } else {
        // the prune bound did not certify the draw (probability ~1e-9): this warp evaluates every kept
        // token of the row from global memory
        path |= PATH_FALLBACK;
        const ArgMax fb = control_fallback_draw<T>(p.x + (int64_t)row * p.ld * ES, n, xP, cut < 0 ? kAllIndex : cut, M,
                                                   invT, rid, st, sd);
        out_token = fb.idx;
        out_s = fb.s;
      }
      if (lane == 0) {
        int st_code = VSAMP_OK;
        if (out_token >= 0 && (int64_t)out_token < n) {
          p.token[row] = out_token;
          if (p.logprob) p.logprob[row] = fminf(out_s - logS, 0.f);
        } else {
          st_code = VSAMP_ERR_INVALID_ARG;
          p.token[row] = -1;
          if (p.logprob) p.logprob[row] = __int_as_float(0x7FC00000);
        }
        if (p.row_status) p.row_status[row] = st_code;
        if (p.stats) {
          p.stats[row * 4 + 0] = passes;
          p.stats[row * 4 + 1] = rounds;
          p.stats[row * 4 + 2] = (int32_t)kept;
          p.stats[row * 4 + 3] = path;
        }
      }
    }
  }
  // no CTA may leave while a peer can still read or write its shared memory
  cg::this_cluster().sync();
}

}  // namespace vsamp
