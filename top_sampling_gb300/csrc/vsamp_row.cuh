// The per-row sampling engine: one thread-block cluster of C CTAs owns one row; each CTA holds a slice
// of the row in shared memory (bulk-copied from HBM once) and every later pass reads shared memory.
//
// Passes (each thread owns q consecutive 16-byte vectors of its CTA's slice, in index order):
//   load   -- cp.async.bulk of each warp's region of the slice on the warp's own mbarrier; a warp
//             re-arms its region with the cluster's next row as soon as its last pass is done;
//   P1     -- row maximum M and a non-finite check;
//   P2     -- S = sum exp((x - M)/T) in 64-bit fixed point, each thread's count of maxima and, when
//             min-p is on, the min-p statistics;
//   select -- top-k / top-p cut: directly inside the maximum's tie group when it holds the cut,
//             otherwise by cluster-wide radix rounds over the order-preserving keys with count and
//             fixed-point mass histograms exchanged through distributed shared memory;
//   ties   -- the cut takes the lowest-index elements of its key group: from per-thread counts and an
//             index-ordered prefix over threads and CTAs, every thread derives its own last kept index
//             (only the thread holding the boundary rescans its chunk);
//   P4     -- Philox4x32-10 per group of four tokens, Gumbel-max over the kept prefix with a prune
//             bound from the kept mass; the CTAs' partial arg-maxes meet in CTA 0's shared memory and
//             the last CTA to arrive reduces them and writes the row's outputs.
// Per-row scalar decisions are computed redundantly, in the same order, by every thread from
// cluster-reduced values (a per-thread `Plan`), so no broadcast barrier is needed for them. Every
// branch that decides which cluster barriers run depends only on cluster-reduced values, so all CTAs
// of a cluster execute the same barrier sequence.
#pragma once

#include "vsamp_device.cuh"
#include "vsamp.h"

namespace vsamp {

enum Mode : int {
  MODE_LSE = 1,       // row_max / row_logsum
  MODE_SELECT = 2,    // stand-alone top-k select (out_idx)
  MODE_CUT = 4,       // cut descriptor
  MODE_MASK = 8,      // uint8 mask of the cut
  MODE_SAMPLE = 16,   // Gumbel-max draw + log-probability
  MODE_LOGPROB = 32,  // log-probability of given tokens (statistics recomputed)
  MODE_TOPN = 64,     // the k_max best tokens (out_idx, ascending index order): the top-k cut, any temperature
  MODE_KEPT = 128,    // log-probability of given tokens renormalised over the cut's kept set (-inf outside it)
};

// Path flags reported in stats[r][3].
enum PathFlag : int {
  PATH_MAXGROUP = 1,    // the cut lies in the maximum's tie group (no radix rounds)
  PATH_RADIX_K = 2,     // top-k radix rounds ran
  PATH_RADIX_P = 4,     // top-p radix rounds ran
  PATH_MINP = 8,        // min-p gave the shortest prefix
  PATH_FALLBACK = 16,   // the prune bound did not certify the draw; all kept tokens were evaluated
  PATH_NOTMA = 32,      // rows were loaded with plain loads (unaligned)
};

struct Params {
  const unsigned char* x;   // [B, ld] elements
  int64_t B, V, ld;         // V: row length (max length when `lengths` is given)
  const int32_t* lengths;
  const float* temperature;
  const int32_t* top_k;
  const float* top_p;
  const float* min_p;
  const uint64_t* seed;
  const uint64_t* step;
  const uint32_t* row_id;
  const int32_t* token_in;
  const int32_t* k_sel;
  int32_t k_max;
  float* row_max;
  float* row_logsum;
  int32_t* out_idx;
  vsamp_cut* cut;
  uint8_t* mask;
  int32_t* token;
  float* logprob;
  int32_t* row_status;
  int32_t* stats;
  int64_t row0;             // first row of this launch
  int32_t q;                // 16-byte vectors per thread
  int32_t tma;              // rows are 16-byte aligned: bulk copies
  long long wait_cycles;    // bound of every device-side wait on a row's load
  int32_t drop_loads;       // failure-detection test hook: loads are armed but never issued, so every
                            // load wait runs out and the rows report VSAMP_ERR_TIMEOUT
  int32_t nbuf;             // slice buffers per CTA (vsamp_sample: 2 streams the next row during this one)
  int32_t vbytes;           // vsamp_sample: a byte per vector after the slices (the largest value bin it holds)
  int64_t v0;               // global index of a row's first element: a vocabulary shard's offset (0 otherwise)
};

constexpr int32_t kNoIndex = -1;
constexpr int32_t kAllIndex = 0x7FFFFFFF;
constexpr float kTwoM32 = 2.3283064365386963e-10f;   // 2^-32
constexpr float kTwoM33 = 1.1641532182693481e-10f;   // 2^-33

// ------------------------------------------------------------------------------------------------
// Element traits: fp32 (4 per vector, 32-bit radix keys) and bf16 (8 per vector, 16-bit radix keys).
// ------------------------------------------------------------------------------------------------
template <typename T>
struct Traits;

template <>
struct Traits<float> {
  static constexpr int VE = 4;
  static constexpr int KB = 32;
  static constexpr int ESIZE = 4;
  __device__ static __forceinline__ void values(const uint4& v, float (&x)[4]) {
    x[0] = __uint_as_float(v.x); x[1] = __uint_as_float(v.y);
    x[2] = __uint_as_float(v.z); x[3] = __uint_as_float(v.w);
  }
  __device__ static __forceinline__ uint32_t rkey_of_value(float x) { return key_f32_bits(__float_as_uint(x)); }
  // every element of the vector is >= xv
  __device__ static __forceinline__ bool all_ge(const uint4& v, float xv) {
    return fminf(fminf(__uint_as_float(v.x), __uint_as_float(v.y)), fminf(__uint_as_float(v.z), __uint_as_float(v.w))) >= xv;
  }
  __device__ static __forceinline__ uint32_t key32(uint32_t rk) { return rk; }
  __device__ static __forceinline__ float value_of_rkey(uint32_t rk) { return value_of_key32(rk); }
  __device__ static __forceinline__ float load_global(const unsigned char* p, int64_t e) {
    return reinterpret_cast<const float*>(p)[e];
  }
};

template <>
struct Traits<__nv_bfloat16> {
  static constexpr int VE = 8;
  static constexpr int KB = 16;
  static constexpr int ESIZE = 2;
  __device__ static __forceinline__ void values(const uint4& v, float (&x)[8]) {
    x[0] = __uint_as_float(v.x << 16); x[1] = __uint_as_float(v.x & 0xFFFF0000u);
    x[2] = __uint_as_float(v.y << 16); x[3] = __uint_as_float(v.y & 0xFFFF0000u);
    x[4] = __uint_as_float(v.z << 16); x[5] = __uint_as_float(v.z & 0xFFFF0000u);
    x[6] = __uint_as_float(v.w << 16); x[7] = __uint_as_float(v.w & 0xFFFF0000u);
  }
  __device__ static __forceinline__ uint32_t rkey_of_value(float x) { return key_bf16_bits(__float_as_uint(x) >> 16); }
  __device__ static __forceinline__ __nv_bfloat162 pair(uint32_t w) {
    __nv_bfloat162 r;
    __builtin_memcpy(&r, &w, 4);
    return r;
  }
  // every element of the vector is >= xv (packed minimum of the eight values)
  __device__ static __forceinline__ bool all_ge(const uint4& v, float xv) {
    const __nv_bfloat162 m = __hmin2(__hmin2(pair(v.x), pair(v.y)), __hmin2(pair(v.z), pair(v.w)));
    return __hbge2(m, __float2bfloat162_rn(xv));      // xv is a bf16 value: the conversion is exact
  }
  __device__ static __forceinline__ uint32_t key32(uint32_t rk) { return key32_of_key16(rk); }
  __device__ static __forceinline__ float value_of_rkey(uint32_t rk) { return value_of_key32(key32_of_key16(rk)); }
  __device__ static __forceinline__ float load_global(const unsigned char* p, int64_t e) {
    const uint32_t h = reinterpret_cast<const uint16_t*>(p)[e];
    return __uint_as_float(h << 16);
  }
};

// ------------------------------------------------------------------------------------------------
// Shared memory.
// ------------------------------------------------------------------------------------------------
struct Mail {             // one CTA's contribution to a cluster exchange (read by peers via DSMEM)
  float f[4];
  uint32_t u[8];
  unsigned long long q[4];
  int32_t i[4];
};

// A cut: the kept prefix ends inside the key group `rk` after `need` of its elements (index order).
struct Cut {
  uint32_t rk;
  unsigned long long above;     // elements with a larger key
  unsigned long long need;      // elements taken from the group
  unsigned long long cnt_eq;    // group size (0 if unknown)
  unsigned long long mass;      // fixed-point mass of the kept prefix
  int whole;                    // every element of the group is kept
  __host__ __device__ unsigned long long kept() const { return above + need; }
};

// Per-row scalar decisions; every thread derives the same values from cluster-reduced statistics.
struct Plan {
  int status;
  int ck_mode;                  // top-k: 0 off, 1 inside the maximum's group, 2 radix
  int cp_mode;                  // top-p: 0 off, 1 inside the maximum's group, 2 radix
  int path;
  float goal_p;                 // top-p radix goal as a fraction of the row mass (< 0: use cp_goal)
  unsigned long long cp_goal;
  Cut ck, cp, fin;
  uint32_t kmin32;              // min-p: keep keys >= kmin32 (fp32 key space)
  int all_cand;                 // P4: evaluate every kept token
  uint32_t bk;                  // P4: a token is a candidate only if its Philox word is < bk
  float kappa;                  // P4: e^3 / kept mass
  float b0;                     // P4: prune bound -log(kappa)
  float logS;                   // log of the row mass (fixed-point units removed)
};

template <int NT>
struct Smem {
  static constexpr int NW = NT / 32;
  unsigned long long bar[NT / 32];   // one mbarrier per warp: its region of the slice has landed
  Mail mail[2];
  // per-warp exchange slots (P1: max, min, flags; P2: mass, counts), double-buffered by exchange parity;
  // every warp of the cluster reads every slot after the cluster barrier
  uint4 ws[2][NT / 32][2];
  // P4 arg-max, per row parity: each warp's partial (its CTA's last warp reduces them), each CTA's
  // partial in CTA 0's copy (the cluster's last warp reduces them), and the two arrival counters
  uint4 apart[2][NT / 32];
  uint4 aslot[2][16];
  uint32_t lcnt[2];
  uint32_t acnt[2];
  uint32_t hcnt[2][256];
  unsigned long long hm[2][256];   // fixed-point mass histograms (64-bit shared-memory adds)
  uint32_t gcnt[256];
  unsigned long long gmass[256];
  uint32_t kmm[2][2];   // radix key rounds: smallest and largest matching key of this CTA, per round parity
  uint32_t gkm[2];      // ... and of the cluster
  uint32_t km_ok;       // this row's km masks are valid, for keys at or above km_rk
  uint32_t km_rk;
  uint32_t tcount[NT];
  uint32_t tpre[NT];
  float wf[NW][3];
  uint32_t wu[NW][4];
  unsigned long long wq[NW][3];
  int32_t wi[NW][2];
  uint32_t bu[8];
  unsigned long long bq[4];
  int32_t bi[4];
  float bf[4];
};

template <int NT>
__host__ __device__ constexpr int slice_offset() {
  return (int)((sizeof(Smem<NT>) + 127) / 128 * 128);
}

// Result of a cluster-wide radix search.
struct RadixOut {
  uint32_t rk;                  // the group's radix key
  unsigned long long cnt_above; // elements with a larger key
  unsigned long long mass_above;
  unsigned long long cnt_eq;    // elements with exactly this key
  unsigned long long mass_eq;
  unsigned long long goal;      // the goal left inside the group (top-p: target mass minus mass above)
  int ok;
  int vsel;                     // sampling kernel: the value bin its first round selected (-1: no value round)
};

// ------------------------------------------------------------------------------------------------
// Value bins of a radix search's first round: 256 bins linear in the value over [xlo, xhi] (the range of the
// candidate values), so that rows whose values share their top key bits (one binade, a narrow distribution,
// a few levels) still spread over many bins and their histogram updates over many addresses. The bin is a
// monotone function of x (a rounded subtraction, a rounded product, a truncation), so the elements of one bin
// are exactly the keys of a contiguous range, which bisection on the same function finds; the later rounds
// refine that range by key bytes, from its highest differing bit down.
// ------------------------------------------------------------------------------------------------
struct ValueBins {
  float xlo, sc;   // bin(x) = min(255, (int)((x - xlo) * sc)); sc == 0: the first round uses key bytes
};

__device__ __forceinline__ ValueBins make_value_bins(float xlo, float xhi) {
  ValueBins vb{xlo, 0.f};
  const float span = __fsub_rn(xhi, xlo);
  if (span > 0.f && span <= 3.0e38f) {
    const float sc = __fdiv_rn(256.f, span);
    if (sc <= 3.0e38f) vb.sc = sc;
  }
  return vb;
}

// The integer part of t in (0, 255) comes from adding 2^23 with rounding toward zero (the sum's unit is 1)
// instead of a float-to-integer conversion, which this part executes at a few results per clock per SM.
__device__ __forceinline__ int value_bin(float x, const ValueBins& vb) {
  const float t = __fmul_rn(__fsub_rn(x, vb.xlo), vb.sc);
  const int ti = (int)(__float_as_uint(__fadd_rz(t, 8388608.0f)) - 0x4B000000u);
  return t >= 255.f ? 255 : (t > 0.f ? ti : 0);
}

// The smallest radix key k in [a, b] whose value falls in a value bin >= target (b + 1 if there is none).
// Called by a full warp: every step tests 32 evenly spaced keys of the interval at once (value_bin is
// monotone in the key), so a 32-bit range takes at most 7 steps.
template <typename Tr>
__device__ __forceinline__ uint32_t first_key_of_bin(uint32_t a, uint32_t b, int target, const ValueBins& vb) {
  const unsigned long long lane = threadIdx.x & 31;
  unsigned long long lo = a, hi = (unsigned long long)b + 1ull;   // the answer lies in [lo, hi]
#pragma unroll 1
  while (lo < hi) {
    const unsigned long long span = hi - lo;   // keys lo .. hi - 1 are untested
    const unsigned long long k = lo + ((span * lane) >> 5);
    const uint32_t bal = __ballot_sync(0xFFFFFFFFu, value_bin(Tr::value_of_rkey((uint32_t)k), vb) >= target);
    if (bal & 1u) return (uint32_t)lo;         // lane 0 tested lo itself
    if (bal == 0u) {                           // every tested key is below the bin: past the last one
      lo += ((span * 31ull) >> 5) + 1ull;
      continue;
    }
    const unsigned long long f = (unsigned long long)(__ffs(bal) - 1);   // >= 1
    hi = lo + ((span * f) >> 5);               // passes
    lo = lo + ((span * (f - 1ull)) >> 5) + 1ull;   // the key before it fails
  }
  return (uint32_t)lo;
}

// The radix rounds after a value-bin round: the key range [klo, khi] of the selected bin, and the first key
// round (the byte holding the highest bit where klo and khi differ) with its prefix.
struct KeyRange {
  uint32_t klo, khi;
  int shift;         // first key round's shift; -1: the bin holds a single key
  uint32_t prefix;   // key bits above the first round's byte (shared by every key of the range)
};

template <typename Tr>
__device__ __forceinline__ KeyRange key_range_of_bin(int b, uint32_t kxlo, uint32_t kxhi, const ValueBins& vb) {
  KeyRange r;
  r.klo = first_key_of_bin<Tr>(kxlo, kxhi, b, vb);
  r.khi = b >= 255 ? kxhi : first_key_of_bin<Tr>(kxlo, kxhi, b + 1, vb) - 1u;
  const uint32_t d = r.klo ^ r.khi;
  if (d == 0u) {
    r.shift = -1;
    r.prefix = r.klo;
  } else {
    r.shift = (31 - __clz((int)d)) & ~7;
    r.prefix = r.shift + 8 >= 32 ? 0u : (r.klo & (0xFFFFFFFFu << (r.shift + 8)));
  }
  return r;
}

// A radix search's first round over every vector of a thread's chunk, in value bins with no floor, counts
// only: one shared-memory atomic per element, and each vector's largest bin into vbyte (when given).
template <typename T, int NTD>
static __device__ __noinline__ void value_round_full(const uint4* mine, int thr_n, ValueBins vb, uint32_t* hc,
                                                     unsigned char* vbyte, int td) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  const int nfull = thr_n / VE;
  auto bins = [&](const uint4 v, int j, int cnt) {
    float x[VE];
    Tr::values(v, x);
    uint32_t vmax = 0u;
#pragma unroll
    for (int i = 0; i < VE; ++i) {
      if (i < cnt) {
        const uint32_t b = (uint32_t)value_bin(x[i], vb);
        vmax = max(vmax, b);
        atomicAdd(&hc[b], 1u);
      }
    }
    if (vbyte) vbyte[j * NTD + td] = (unsigned char)vmax;
  };
  int j = 0;
  for (; j + 2 <= nfull; j += 2) {
    const uint4 v0 = mine[j], v1 = mine[j + 1];
    bins(v0, j, VE);
    bins(v1, j + 1, VE);
  }
  for (; j < nfull; ++j) bins(mine[j], j, VE);
  if (nfull * VE < thr_n) bins(mine[nfull], nfull, thr_n - nfull * VE);
}

template <typename T, int NT, int MODE>
struct RowEngine {
  using Tr = Traits<T>;
  static constexpr int VE = Tr::VE;
  static constexpr int NW = NT / 32;

  const Params& p;
  Smem<NT>& sh;
  const uint4* mine;       // this thread's vectors in shared memory
  cg::cluster_group cluster;
  int C, crank, row, t, lane, warp, q;
  int64_t n;               // valid elements in the row
  int64_t thr_e0;          // global index of this thread's first element
  int thr_n;               // valid elements in this thread's chunk
  int xc;                  // cluster exchange counter (ping-pong parity)
  int passes, rounds;

  __device__ RowEngine(const Params& p_, Smem<NT>& sh_)
      : p(p_), sh(sh_), cluster(cg::this_cluster()) {
    C = gridDim.x;
    crank = blockIdx.x;
    row = 0;
    t = threadIdx.x;
    lane = t & 31;
    warp = t >> 5;
    q = p.q;
    mine = nullptr;
    xc = 0;
    passes = 0;
    rounds = 0;
  }
  // After the slice, where the launch has room (p.vbytes): byte j * NT + t, the largest value bin of vector j of
  // this thread's chunk in the last value round; then four words per thread, word f * NT + t: vm (f = 0, 1: the
  // vectors with such a byte, those that matched that round) and km (f = 2, 3: the vectors holding a key at or
  // above sh.km_rk, set by mass_above_key). Kept in shared memory so they hold no registers outside the radix
  // searches.
  __device__ __forceinline__ unsigned char* vbyte() const {
    return p.vbytes ? reinterpret_cast<unsigned char*>(&sh) + slice_offset<NT>() + (size_t)NT * p.q * 16 : nullptr;
  }
  __device__ __forceinline__ uint32_t& vmk(int f) const {
    return reinterpret_cast<uint32_t*>(vbyte() + ((size_t)NT * p.q + 15) / 16 * 16)[f * NT + t];
  }
  __device__ __forceinline__ bool masked() const { return (thr_n + VE - 1) / VE <= 64; }
  // m reduced to the vectors whose largest bin in the last value round is at or above vsel
  __device__ void by_bin(uint32_t (&m)[2], int vsel) const {
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      uint32_t o = 0u;
      for (uint32_t bits = m[w]; bits; bits &= bits - 1u) {
        const int b = __ffs(bits) - 1;
        if ((int)vbyte()[(w * 32 + b) * NT + t] >= vsel) o |= 1u << b;
      }
      m[w] = o;
    }
  }
  // this thread's vectors: warp w's region of the slice starts at vector w * 32 * qmax (the launch's q); a row
  // spread over fewer vectors per thread (qr <= qmax) fills the first 32 * qr vectors of it, qr per lane
  __device__ void set_slice(const unsigned char* slice, int qmax) {
    mine = reinterpret_cast<const uint4*>(slice) + (size_t)warp * 32 * qmax + (size_t)lane * q;
  }

  // ---------------- cluster exchange primitives ----------------
  __device__ __forceinline__ Mail& my_mail() { return sh.mail[xc & 1]; }
  // All threads, after this CTA's mail is written (by thread 0): publishes it and waits for the peers
  // (for a one-CTA cluster, a block barrier). Mail is double-buffered by the exchange parity, so the
  // peers' copies may be read until the next exchange.
  __device__ __forceinline__ void exchange() {
    if (C == 1) __syncthreads();
    else cluster_barrier_shared();
  }
  __device__ __forceinline__ const Mail* peer_mail(int rank) {
    return cluster.map_shared_rank(&sh.mail[xc & 1], rank);
  }
  __device__ __forceinline__ void exchange_done() { ++xc; }
  // slot k of warp w of CTA r in the current exchange's slots (after exchange())
  __device__ __forceinline__ uint4 wslot(int r, int w, int k) {
    const uint4* a = &sh.ws[xc & 1][w][k];
    return C == 1 ? *a : dsmem_load_v4(dsmem_map(a, (uint32_t)r));
  }

  // Exclusive scan of tcount[] over threads (index order) into tpre[]; returns the block total.
  __device__ uint32_t block_scan_tcount() {
    __syncthreads();
    const uint32_t v = sh.tcount[t];
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) sh.wu[warp][1] = incl;
    __syncthreads();
    uint32_t wbase = 0, total = 0;
#pragma unroll
    for (int w = 0; w < NW; ++w) {
      const uint32_t s = sh.wu[w][1];
      if (w < warp) wbase += s;
      total += s;
    }
    sh.tpre[t] = wbase + incl - v;
    __syncthreads();
    return total;
  }

  // Calls f(global index, value) for every valid element of this thread's chunk, in index order.
  template <class F>
  __device__ __forceinline__ void for_each(F&& f) {
    const int nfull = thr_n / VE;
    for (int j = 0; j < nfull; ++j) {
      float x[VE];
      Tr::values(mine[j], x);
#pragma unroll
      for (int i = 0; i < VE; ++i) f(thr_e0 + (int64_t)j * VE + i, x[i]);
    }
    const int tail = thr_n - nfull * VE;
    if (tail) {
      float x[VE];
      Tr::values(mine[nfull], x);
#pragma unroll
      for (int i = 0; i < VE; ++i)
        if (i < tail) f(thr_e0 + (int64_t)nfull * VE + i, x[i]);
    }
  }

  // Calls f(global index, value) -> bool for every valid element of the vectors of this thread's chunk whose
  // bit is set in cand (bit b of word w: vector 32 w + b), in index order; out gets the bits of the vectors
  // where f returned true for some element.
  template <class F>
  __device__ __forceinline__ void for_each_cand(const uint32_t (&cand)[2], uint32_t (&out)[2], F&& f) {
    for_each_cand(cand, out, f, [](int) {});
  }
  // the same, with g(vector) called after each vector
  template <class F, class Gv>
  __device__ __forceinline__ void for_each_cand(const uint32_t (&cand)[2], uint32_t (&out)[2], F&& f, Gv&& g) {
#pragma unroll
    for (int w = 0; w < 2; ++w) {
      uint32_t bits = cand[w], hit = 0u;
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1u;
        const int j = w * 32 + b;
        const int cnt = thr_n - j * VE < VE ? thr_n - j * VE : VE;
        float x[VE];
        Tr::values(mine[j], x);
        bool any = false;
#pragma unroll
        for (int i = 0; i < VE; ++i)
          if (i < cnt && f(thr_e0 + (int64_t)j * VE + i, x[i])) any = true;
        g(j);
        if (any) hit |= 1u << b;
      }
      out[w] = hit;
    }
  }

  // Cluster exclusive prefix of a per-CTA value: returns (sum over lower ranks, total) to every thread.
  __device__ void cluster_prefix_u32(uint32_t mine_val, int slot, uint32_t& pre, uint32_t& total) {
    if (t == 0) my_mail().u[slot] = mine_val;
    exchange();
    // every warp reads the peers' values (no broadcast barrier)
    const uint32_t v = lane < C ? peer_mail(lane)->u[slot] : 0u;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
      if (lane >= o) incl += y;
    }
    total = __shfl_sync(kFullMask, incl, 31);
    pre = __shfl_sync(kFullMask, incl - v, crank);
    exchange_done();
  }

  // Fixed-point mass (as the radix histograms sum it) of the row's keys above rk0, summed over the cluster.
  // Collective over the cluster; one exchange. vsel >= 0: the value bin of rk0 in the last value round, whose
  // bytes limit the pass to the vectors reaching it. Records km (the vectors holding a key >= rk0).
  __device__ unsigned long long mass_above_key(uint32_t rk0, float M, float c1, int vsel) {
    unsigned long long s = 0ull;
    if (p.vbytes && masked()) {
      const int nvec = (thr_n + VE - 1) / VE;
      uint32_t v[2];
      v[0] = nvec >= 32 ? 0xFFFFFFFFu : ((1u << nvec) - 1u);
      v[1] = nvec >= 64 ? 0xFFFFFFFFu : (nvec > 32 ? ((1u << (nvec - 32)) - 1u) : 0u);
      if (vsel >= 0) {
        v[0] = vmk(0);
        v[1] = vmk(1);
        by_bin(v, vsel);
      }
      uint32_t o[2];
      for_each_cand(v, o, [&](int64_t, float x) -> bool {
        const uint32_t rk = Tr::rkey_of_value(x);
        if (rk > rk0) s += mass_fx(ex2_approx((x - M) * c1));
        return rk >= rk0;
      });
      vmk(2) = o[0];
      vmk(3) = o[1];
      if (t == 0) {
        sh.km_ok = 1u;   // every thread of every CTA reaches this point (read after the exchange below)
        sh.km_rk = rk0;
      }
    } else {
      for_each([&](int64_t, float x) {
        if (Tr::rkey_of_value(x) > rk0) s += mass_fx(ex2_approx((x - M) * c1));
      });
    }
    ++passes;
    s = warp_sum_u64(s);
    if (lane == 0) sh.ws[xc & 1][warp][0] = make_uint4((uint32_t)s, (uint32_t)(s >> 32), 0u, 0u);
    exchange();
    unsigned long long a = 0ull;
    for (int i = lane; i < C * NW; i += 32) {
      const uint4 v = wslot(i / NW, i % NW, 0);
      a += ((unsigned long long)v.y << 32) | v.x;
    }
    a = warp_sum_u64(a);
    exchange_done();
    return a;
  }

  // Per-thread count of elements equal to xv, into tcount[].
  __device__ void count_equal_pass(float xv) {
    uint32_t c = 0;
    if (sh.km_ok && Tr::rkey_of_value(xv) >= sh.km_rk && masked()) {   // only the vectors holding such a key
      uint32_t o[2];
      const uint32_t km[2] = {vmk(2), vmk(3)};
      for_each_cand(km, o, [&](int64_t, float x) -> bool {
        c += (x == xv) ? 1u : 0u;
        return false;
      });
    } else {
      for_each([&](int64_t, float x) { c += (x == xv) ? 1u : 0u; });
    }
    sh.tcount[t] = c;
    ++passes;
  }

  // The group of value xv keeps its `need` lowest-index elements. tcount[]/tpre[] hold each thread's
  // count of the group and its exclusive prefix in the CTA; cpre is the count over lower CTA ranks.
  // Returns this thread's last kept index (kAllIndex: every element of the group in its chunk is kept;
  // kNoIndex: none). The thread holding the need-th element gets it in `boundary`; its warp finds it
  // together (one 16-byte vector of that thread's chunk per lane, then a warp prefix of the counts).
  // start: elements equal to xv before this thread's chunk (index order); cnt: those in its chunk
  __device__ int32_t local_cut_index(float xv, unsigned long long need, unsigned long long start,
                                     unsigned long long cnt, int32_t& boundary) {
    boundary = kNoIndex;
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
          for (int i = 0; i < VE; ++i) c += (j * VE + i < src_n && x[i] == xv) ? 1u : 0u;
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
          for (int i = 0; i < VE; ++i) {
            if (idx < 0 && j * VE + i < src_n && x[i] == xv && ++seen == remaining)
              idx = (int32_t)(src_e0 + (long long)j * VE + i);
          }
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
        return found;
      }
    }
    if (start >= need) return kNoIndex;
    return kAllIndex;
  }

  // ---------------- radix search ----------------
  // COUNT (mass_mode == false): the group holding the goal-th largest element (1-based).
  // MASS: the group where the cumulative mass (from the largest key down) first reaches the goal;
  //       if goal_p >= 0 the goal is ceil(goal_p * total mass of the row) taken in the first round.
  // want_mass: also histogram masses (mass_above / mass_eq are valid).
  // floor_rk: keys below it are left out of the histograms. The caller passes a floor only when the goal is
  //   reached within the keys at or above it, so the group found and its counts do not change.
  // xmin: the row's smallest value. When the candidates span a finite range, the first round bins values
  //   linearly over it (ValueBins) and the key rounds then refine the selected bin's key range; otherwise the
  //   rounds take the key bytes from the top.
  // Each round visits only the vectors of the thread's chunk that held an element matching the previous
  // round's prefix (chunks of at most 64 vectors; longer chunks visit every vector).
  __device__ RadixOut radix_search(bool mass_mode, unsigned long long goal, float goal_p, bool want_mass, float M,
                                   float c1, uint32_t floor_rk, float xmin) {
    RadixOut out{};
    out.ok = 1;
    out.vsel = -1;
    uint32_t prefix = 0;
    unsigned long long cnt_above = 0, mass_above = 0;
    const bool hist_mass = want_mass || mass_mode;
    const int nvec = (thr_n + VE - 1) / VE;
    const bool masked = nvec <= 64;
    uint32_t cand[2];
    cand[0] = nvec >= 32 ? 0xFFFFFFFFu : ((1u << nvec) - 1u);
    cand[1] = nvec >= 64 ? 0xFFFFFFFFu : (nvec > 32 ? ((1u << (nvec - 32)) - 1u) : 0u);
    bool all = true;   // cand holds every vector
    if (masked && floor_rk && sh.km_ok && floor_rk >= sh.km_rk) {   // keys at or above the floor lie in the km vectors
      cand[0] = vmk(2);
      cand[1] = vmk(3);
      all = false;
    }
    int vsel_next = -1;   // the round after a value round: the vectors reaching the selected bin
    // the candidates' value range: [max(xmin, value of floor_rk), M]
    const float xlo = floor_rk ? fmaxf(xmin, Tr::value_of_rkey(floor_rk)) : xmin;
    const ValueBins vb = make_value_bins(xlo, M);
    bool vround = vb.sc > 0.f;          // this round bins values
    bool first = true;
    uint32_t klo = 0u, khi = 0xFFFFFFFFu;
    int shift = vround ? 0 : Tr::KB - 8;
    for (;;) {
      const int par = xc & 1;
      uint32_t* hc = sh.hcnt[par];
      unsigned long long* hm = sh.hm[par];
      for (int b = t; b < 256; b += NT) { hc[b] = 0; hm[b] = 0ull; }
      if (t == 0) { sh.kmm[par][0] = 0xFFFFFFFFu; sh.kmm[par][1] = 0u; }
      __syncthreads();
      // the first key round after a value round also finds the smallest and largest matching key: when they
      // are equal (a bin holding one distinct value) the search ends there
      const bool track = vsel_next >= 0;
      if (vsel_next >= 0 && masked && p.vbytes) {
        by_bin(cand, vsel_next);
        all = false;
      }
      vsel_next = -1;
      const int hi_shift = shift + 8;
      const uint32_t hmask = hi_shift >= 32 ? 0u : (0xFFFFFFFFu << hi_shift);
      uint32_t run_bin = 0xFFFFFFFFu, run_cnt = 0;
      unsigned long long run_mass = 0;
      auto flush = [&]() {
        if (run_cnt) {
          atomicAdd(&hc[run_bin], run_cnt);
          if (hist_mass) atomicAdd(&hm[run_bin], run_mass);   // one 64-bit shared-memory add, no return
        }
      };
      uint32_t vmax = 0u;   // a value round: the largest bin of the vector being visited
      uint32_t kmn = 0xFFFFFFFFu, kmx = 0u;   // a key round: the smallest and largest matching key
      auto visit = [&](int64_t, float x) -> bool {
        const uint32_t rk = Tr::rkey_of_value(x);
        const bool match = vround ? rk >= floor_rk
                                  : ((rk & hmask) == (prefix & hmask) && rk >= floor_rk && rk >= klo && rk <= khi);
        if (match && track) {
          kmn = min(kmn, rk);
          kmx = max(kmx, rk);
        }
        if (match && !hist_mass) {
          // a count-only round: one atomic per element, no dependency from one element to the next
          const uint32_t bin = vround ? (uint32_t)value_bin(x, vb) : ((rk >> shift) & 255u);
          vmax = max(vmax, bin);
          atomicAdd(&hc[bin], 1u);
        } else if (match) {
          // a mass round: runs of equal bins merged before the (carry-propagating) 64-bit adds
          const uint32_t bin = vround ? (uint32_t)value_bin(x, vb) : ((rk >> shift) & 255u);
          vmax = max(vmax, bin);
          if (bin != run_bin) {
            flush();
            run_bin = bin;
            run_cnt = 0;
            run_mass = 0;
          }
          ++run_cnt;
          if (hist_mass) run_mass += mass_fx(ex2_approx((x - M) * c1));
        }
        return match;
      };
      if (masked && all && vround && !hist_mass && floor_rk == 0u) {
        // the first round of a count search over the whole chunk
        value_round_full<T, NT>(mine, thr_n, vb, hc, vbyte(), t);
        if (p.vbytes) {
          vmk(0) = cand[0];
          vmk(1) = cand[1];
        }
      } else if (masked) {
        uint32_t next[2];
        unsigned char* const vb8 = vround ? vbyte() : nullptr;
        for_each_cand(cand, next, visit, [&](int j) {
          if (vb8) vb8[j * NT + t] = (unsigned char)vmax;
          vmax = 0u;
        });
        cand[0] = next[0];
        cand[1] = next[1];
        if (vround && p.vbytes) {
          vmk(0) = next[0];
          vmk(1) = next[1];
        }
      } else {
        for_each([&](int64_t e, float x) { (void)visit(e, x); });
      }
      flush();
      if (track) {
        kmn = __reduce_min_sync(kFullMask, kmn);
        kmx = __reduce_max_sync(kFullMask, kmx);
        if (lane == 0) {
          atomicMin(&sh.kmm[par][0], kmn);
          atomicMax(&sh.kmm[par][1], kmx);
        }
      }
      ++passes;
      ++rounds;
      exchange();
      // cluster-sum the histograms
      // four peers' values of a bin are loaded before any is added (one round trip per four ranks)
      for (int b = t; b < 256; b += NT) {
        uint32_t cs = 0;
        unsigned long long ms = 0;
        for (int r0 = 0; r0 < C; r0 += 4) {
          uint32_t cv[4] = {0u, 0u, 0u, 0u};
          unsigned long long mv[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            if (r0 + k < C) {
              cv[k] = dsmem_load_u32(dsmem_map(&sh.hcnt[par][b], (uint32_t)(r0 + k)));
              if (hist_mass) mv[k] = dsmem_load_u64(dsmem_map(&sh.hm[par][b], (uint32_t)(r0 + k)));
            }
          }
#pragma unroll
          for (int k = 0; k < 4; ++k) {
            cs += cv[k];
            ms += mv[k];
          }
        }
        sh.gcnt[b] = cs;
        sh.gmass[b] = ms;
      }
      if (t == 0 && track) {   // the cluster's smallest and largest matching key
        uint32_t mn[16], mx[16];
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          mn[r] = 0xFFFFFFFFu;
          mx[r] = 0u;
          if (r < C) {
            mn[r] = C == 1 ? sh.kmm[par][0] : dsmem_load_u32(dsmem_map(&sh.kmm[par][0], (uint32_t)r));
            mx[r] = C == 1 ? sh.kmm[par][1] : dsmem_load_u32(dsmem_map(&sh.kmm[par][1], (uint32_t)r));
          }
        }
        uint32_t a = 0xFFFFFFFFu, z = 0u;
#pragma unroll
        for (int r = 0; r < 16; ++r) {
          a = min(a, mn[r]);
          z = max(z, mx[r]);
        }
        sh.gkm[0] = a;
        sh.gkm[1] = z;
      }
      exchange_done();
      __syncthreads();
      if (mass_mode && goal_p >= 0.f && first) {
        if (warp == 0) {
          unsigned long long tot = 0;
          for (int b = lane; b < 256; b += 32) tot += sh.gmass[b];
          tot = warp_sum_u64(tot);
          if (lane == 0) sh.bq[3] = ceil_mul_frac(goal_p, tot);
        }
        __syncthreads();
        goal = sh.bq[3];
      }
      first = false;
      // warp 0: suffix scan from the top bin; lane l covers bins 255-8l .. 248-8l
      if (warp == 0) {
        uint32_t lc = 0;
        unsigned long long lm = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int b = 255 - 8 * lane - i;
          lc += sh.gcnt[b];
          lm += sh.gmass[b];
        }
        uint32_t ic = lc;
        unsigned long long im = lm;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t yc = __shfl_up_sync(kFullMask, ic, o);
          const unsigned long long ym = __shfl_up_sync(kFullMask, im, o);
          if (lane >= o) { ic += yc; im += ym; }
        }
        const unsigned long long ec = ic - lc, em = im - lm;   // bins above this lane's
        const unsigned long long g = goal;
        const bool mine_has = mass_mode ? (em < g && g <= im) : (ec < g && g <= (unsigned long long)ic);
        const uint32_t ballot = __ballot_sync(kFullMask, mine_has);
        if (ballot == 0) {
          if (lane == 0) sh.bu[2] = 0xFFFFFFFFu;
        } else if (lane == __ffs(ballot) - 1) {
          unsigned long long ac = ec, am = em;
          int sel = -1;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int b = 255 - 8 * lane - i;
            const unsigned long long c = sh.gcnt[b], m = sh.gmass[b];
            const bool hit = mass_mode ? (am < g && g <= am + m) : (ac < g && g <= ac + c);
            if (hit && sel < 0) sel = b;
            if (sel < 0) { ac += c; am += m; }
          }
          sh.bu[2] = (uint32_t)sel;
          sh.bq[0] = ac;
          sh.bq[1] = am;
        }
      }
      __syncthreads();
      const uint32_t sel = sh.bu[2];
      if (sel > 255u) {   // cannot happen with consistent histograms; reported as an error
        out.ok = 0;
        __syncthreads();
        return out;
      }
      const unsigned long long ac = sh.bq[0], am = sh.bq[1];
      out.cnt_eq = sh.gcnt[sel];
      out.mass_eq = sh.gmass[sel];
      __syncthreads();
      cnt_above += ac;
      mass_above += am;
      if (mass_mode) goal -= am; else goal -= ac;
      if (vround) {
        // the selected bin's key range (every thread bisects the same monotone function)
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
      if (track && sh.gkm[0] == sh.gkm[1]) {   // every matching element holds the same key: the group
        prefix = sh.gkm[0];
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
    return out;
  }
};

// ------------------------------------------------------------------------------------------------
// Perturbed score of one candidate token: E = -log1p(-u) = -log(1 - u), evaluated on the exact side of
// 1/2 (1 - u is itself a cell midpoint of the complementary word ~b), score = s - log(E).
// ------------------------------------------------------------------------------------------------
static __device__ __noinline__ float gumbel_score(float s, uint32_t b) {
  float E;
  if (b < 0x80000000u) {
    const float u = fmaf((float)b, kTwoM32, kTwoM33);
    E = -log1pf(-u);
  } else {
    const float um = fmaf((float)(~b), kTwoM32, kTwoM33);
    E = -logf(um);
  }
  return s - logf(E);
}

// ------------------------------------------------------------------------------------------------
// The two streaming passes over a thread's chunk, kept out of line: the kernel's per-row state is saved
// once around each call and the loop gets the registers (the Philox rounds, their keys) to itself.
// ------------------------------------------------------------------------------------------------
struct MassPart {
  unsigned long long s;     // fixed-point mass of the chunk
  unsigned long long mge;   // min-p: mass of the elements at or above the threshold
  uint32_t cm;              // elements equal to the row maximum
  uint32_t cge;             // min-p: elements at or above the threshold
  uint32_t minkey;          // min-p: smallest such key (fp32 key space)
  uint32_t cmin;            // min-p: its count
};

// P2: sum of 2^((x - M) * c1) in 2^-40 fixed point (each 16-byte vector summed pairwise in a fixed
// order, then converted), the count of maxima and, with MINP, the min-p statistics.
template <typename T, bool MINP>
__device__ __forceinline__ MassPart mass_pass_body(const uint4* mine, int thr_n, float M, float c1, uint32_t kmin32) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  MassPart o{0ull, 0ull, 0u, 0u, 0xFFFFFFFFu, 0u};
  const int nfull = thr_n / VE;
  const float2 mM = make_float2(-M, -M), cc = make_float2(c1, c1);
  uint32_t cm2 = 0;   // bf16: maxima counts in two 16-bit lanes
  auto minp_stats = [&](const float (&x)[VE], const float (&w)[VE], int cnt) {
#pragma unroll
    for (int i = 0; i < VE; ++i) {
      const uint32_t k32 = key_f32_bits(__float_as_uint(x[i]));
      if (i < cnt && k32 >= kmin32) {
        ++o.cge;
        o.mge += mass_fx(w[i]);
        if (k32 < o.minkey) { o.minkey = k32; o.cmin = 1; }
        else if (k32 == o.minkey) ++o.cmin;
      }
    }
  };
  for (int j = 0; j < nfull; ++j) {
    const uint4 v = mine[j];
    float x[VE];
    Tr::values(v, x);
    float2 w2[VE / 2];
#pragma unroll
    for (int h = 0; h < VE / 2; ++h) {
      const float2 e = __fmul2_rn(__fadd2_rn(make_float2(x[2 * h], x[2 * h + 1]), mM), cc);
      w2[h] = make_float2(ex2_approx(e.x), ex2_approx(e.y));
    }
    if constexpr (VE == 8) {
      const __nv_bfloat162 M2 = __float2bfloat162_rn(M);   // M is a bf16 value: exact
      cm2 += __heq2_mask(Tr::pair(v.x), M2) & 0x00010001u;
      cm2 += __heq2_mask(Tr::pair(v.y), M2) & 0x00010001u;
      cm2 += __heq2_mask(Tr::pair(v.z), M2) & 0x00010001u;
      cm2 += __heq2_mask(Tr::pair(v.w), M2) & 0x00010001u;
    } else {
#pragma unroll
      for (int i = 0; i < VE; ++i) o.cm += x[i] == M ? 1u : 0u;
    }
    if (MINP) {
      float w[VE];
#pragma unroll
      for (int h = 0; h < VE / 2; ++h) { w[2 * h] = w2[h].x; w[2 * h + 1] = w2[h].y; }
      minp_stats(x, w, VE);
    }
    // (w0 + w4) + (w2 + w6) and (w1 + w5) + (w3 + w7) for eight, (w0 + w2) and (w1 + w3) for four
    float2 a;
    if constexpr (VE == 8) a = __fadd2_rn(__fadd2_rn(w2[0], w2[2]), __fadd2_rn(w2[1], w2[3]));
    else a = __fadd2_rn(w2[0], w2[1]);
    // bf16: one conversion per eight exponentials leaves the FP64 pipe idle most of the time, so the conversion
    // instruction is cheaper there than mass_fx's arithmetic (both round to nearest-even: the same value)
    if constexpr (VE == 8) o.s += __float2ull_rn((a.x + a.y) * kMassScale);
    else o.s += mass_fx(a.x + a.y);
  }
  const int cnt = thr_n - nfull * VE;
  if (cnt > 0) {
    float x[VE], w[VE];
    Tr::values(mine[nfull], x);
#pragma unroll
    for (int i = 0; i < VE; ++i) {
      const bool ok = i < cnt;
      const float d = x[i] - M;
      w[i] = ok ? ex2_approx(d * c1) : 0.f;
      o.cm += (ok && d == 0.f) ? 1u : 0u;
    }
    if (MINP) minp_stats(x, w, cnt);
#pragma unroll
    for (int h = VE / 2; h >= 1; h >>= 1)
#pragma unroll
      for (int i = 0; i < h; ++i) w[i] += w[i + h];
    o.s += mass_fx(w[0]);
  }
  o.cm += (cm2 & 0xFFFFu) + (cm2 >> 16);
  return o;
}

template <typename T, bool MINP>
static __device__ __noinline__ MassPart mass_pass(const uint4* mine, int thr_n, float M, float c1, uint32_t kmin32) {
  return mass_pass_body<T, MINP>(mine, thr_n, M, c1, kmin32);
}

// The vectors of a thread's chunk that hold a kept token (no Philox words: used when every kept token
// is a candidate, i.e. the kept mass is below e^3).
template <typename T>
static __device__ __noinline__ unsigned long long kept_vectors(const uint4* mine, int thr_n, int64_t thr_e0, float xP,
                                                              int32_t It) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  const int nfull = thr_n / VE;
  const int nvec = (thr_n + VE - 1) / VE;
  unsigned long long m = 0ull;
  for (int j = 0; j < nvec; ++j) {
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

// P4 main pass: one Philox4x32-10 word per kept token (x > xP, or x == xP and index <= It); returns the
// mask of vectors holding a kept token whose word is below bk. Vectors j < jfull whose every element is
// >= xP are kept whole (their indices are <= It).
template <typename T>
static __device__ __noinline__ unsigned long long draw_pass(const uint4* mine, int thr_n, int64_t thr_e0, int jfull,
                                                          float xP, int32_t It, uint32_t g0, uint32_t rid,
                                                          uint32_t st_lo, uint32_t st_hi, PhiloxKey key, uint32_t bk) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  const int nfull = thr_n / VE;
  const int nvec = (thr_n + VE - 1) / VE;
  unsigned long long flagged = 0ull;
  for (int j = 0; j < nvec; ++j) {
    const uint4 v = mine[j];
    uint32_t bmin = 0xFFFFFFFFu;
    if (j < jfull && Tr::all_ge(v, xP)) {
#pragma unroll
      for (int g = 0; g < VE / 4; ++g) {
        const uint4 w4 = philox4x32_10(make_uint4(g0 + (uint32_t)(j * (VE / 4) + g), rid, st_lo, st_hi), key);
        bmin = min(bmin, min(min(w4.x, w4.y), min(w4.z, w4.w)));
      }
    } else {
      float x[VE];
      Tr::values(v, x);
      const int cnt = j < nfull ? VE : thr_n - nfull * VE;
      const int64_t e0 = thr_e0 + (int64_t)j * VE;
      uint32_t gmask = 0u;   // groups of four tokens holding a kept token
#pragma unroll
      for (int i = 0; i < VE; ++i)
        if (i < cnt && (x[i] > xP || (x[i] == xP && e0 + i <= (int64_t)It))) gmask |= 1u << (i >> 2);
      if (!gmask) continue;
#pragma unroll
      for (int g = 0; g < VE / 4; ++g) {
        if (!((gmask >> g) & 1u)) continue;
        const uint4 w4 = philox4x32_10(make_uint4(g0 + (uint32_t)(j * (VE / 4) + g), rid, st_lo, st_hi), key);
        bmin = min(bmin, min(min(w4.x, w4.y), min(w4.z, w4.w)));
      }
    }
    if (bmin < bk) flagged |= 1ull << j;
  }
  return flagged;
}

// ------------------------------------------------------------------------------------------------
// The kernel: persistent clusters. Cluster y handles rows y, y + G, y + 2G, ... (G = gridDim.y); every
// warp bulk-copies its own region of the slice; right after its last pass over row r it copies its region
// of row r + G (the P4 fallback pass, which is rare, then reads the row from global memory), so HBM
// streams while the row's reductions and the other CTAs on the SM finish.
// ------------------------------------------------------------------------------------------------
template <typename T, int NT, int MODE>
__global__ void __launch_bounds__(NT, (NT <= 128 ? 6 : 3)) row_kernel(const Params p) {
  using Tr = Traits<T>;
  using Eng = RowEngine<T, NT, MODE>;
  constexpr int VE = Tr::VE;
  constexpr int ES = Tr::ESIZE;
  constexpr bool kSel = (MODE & MODE_SELECT) != 0;
  constexpr bool kTopn = (MODE & MODE_TOPN) != 0;
  constexpr bool kCutLike = (MODE & (MODE_CUT | MODE_SAMPLE | MODE_TOPN | MODE_KEPT)) != 0;
  extern __shared__ __align__(128) unsigned char dyn[];
  Smem<NT>& sh = *reinterpret_cast<Smem<NT>*>(dyn);
  unsigned char* slice = dyn + slice_offset<NT>();
  Eng E(p, sh);
  Plan plan{};          // per-row decisions, computed identically by every thread
  const int t = E.t, lane = E.lane, warp = E.warp, q = E.q, C = E.C, crank = E.crank;
  const int64_t G = gridDim.y;
  const int64_t first = blockIdx.y;
  const int64_t warp_region = (int64_t)32 * q * 16;    // each warp's region of the slice (bytes)

  auto row_len = [&](int64_t r) -> int64_t {
    int64_t n = p.V;
    if (p.lengths) n = p.lengths[r];
    return (n > 0 && n <= p.V) ? n : 0;
  };
  // vectors per thread for a row of n elements: q, or for rows of their own lengths (a ragged batch) the fewest
  // (odd, for conflict-free 16-byte loads) that spread the row over every CTA of the cluster
  auto q_of = [&](int64_t n) -> int {
    if (!p.lengths) return q;
    const int64_t nv = (n + VE - 1) / VE;
    int64_t qq = (nv + (int64_t)C * NT - 1) / ((int64_t)C * NT);
    if (qq < 1) qq = 1;
    if ((qq & 1) == 0 && qq < q) ++qq;
    return (int)(qq < q ? qq : q);
  };
  // lane 0 of each warp: bulk copy of the warp's part of row r (its 16-byte-aligned part) into the warp's
  // region; returns whether a copy is in flight
  auto issue_warp = [&](int64_t r) -> bool {
    const int64_t n = row_len(r);
    const int qr = q_of(n);
    const int64_t span = (int64_t)NT * qr * VE, e0 = (int64_t)crank * span;
    const int64_t c = n - e0 < 0 ? 0 : (n - e0 > span ? span : n - e0);
    const int64_t b16 = (c * ES) & ~(int64_t)15;
    const int64_t wb = (int64_t)32 * qr * 16, lo = (int64_t)warp * wb;
    int64_t nb = b16 - lo;
    nb = nb < 0 ? 0 : (nb > wb ? wb : nb);
    mbar_arrive_expect_tx(&sh.bar[warp], (uint32_t)nb);
    if (nb && !p.drop_loads) {
      bulk_copy_g2s(slice + (int64_t)warp * warp_region, p.x + ((int64_t)r * p.ld + e0) * ES + lo, (uint32_t)nb,
                    &sh.bar[warp]);
      return true;
    }
    return false;
  };
  if (t == 0) { sh.acnt[0] = 0u; sh.acnt[1] = 0u; sh.lcnt[0] = 0u; sh.lcnt[1] = 0u; }
  int uses = 0;            // completed phases of this warp's mbarrier
  bool pending = false;    // this warp's mbarrier has an armed phase that has not completed
  bool inflight = false;   // lane 0: a bulk copy into this warp's region may still be landing
  if (p.tma) {
    if (lane == 0) {
      mbar_init(&sh.bar[warp], 1);
      fence_mbar_init();
    }
    __syncthreads();
    if (first < p.B) {
      if (lane == 0) inflight = issue_warp(first);
      pending = true;
    }
  }
  bool dead = false;   // a load timed out: later rows are reported as timed out, not computed

  for (int64_t k = 0;; ++k) {
    const int64_t row = first + k * G;
    if (row >= p.B) break;
    E.row = (int)row;
    E.passes = 0;
    E.rounds = 0;
    if (t == 0) sh.km_ok = 0u;   // read only after this row's first cluster exchange

  // ---------------- row geometry ----------------
  int64_t n = p.V;
  if (p.lengths) n = p.lengths[row];
  const bool bad_len = !(n > 0 && n <= p.V);
  if (bad_len) n = 0;
  E.n = n;
  const int qr = q_of(n);
  E.q = qr;
  E.set_slice(slice, q);
  const int64_t elems_cta = (int64_t)NT * qr * VE;
  const int64_t cta_e0 = (int64_t)crank * elems_cta;
  const int64_t cta_n = n - cta_e0 < 0 ? 0 : (n - cta_e0 > elems_cta ? elems_cta : n - cta_e0);
  E.thr_e0 = cta_e0 + (int64_t)t * qr * VE;
  {
    const int64_t r = n - E.thr_e0;
    E.thr_n = r < 0 ? 0 : (r > (int64_t)qr * VE ? qr * VE : (int)r);
  }
  const unsigned char* grow = p.x + ((int64_t)row * p.ld + cta_e0) * ES;
  // slice element of the CTA's element e: thread e / (qr VE), in its warp's region
  auto slice_elem = [&](int64_t e) -> int64_t {
    const int64_t th = e / ((int64_t)qr * VE);
    return ((th >> 5) * 32 * q + (th & 31) * qr) * VE + (e - th * qr * VE);
  };

  // ---------------- the row's parameters (loads issued before the wait, so their latency overlaps it) ----
  float temp = 1.f, topp = 1.f, minp = 0.f;
  int32_t topk = 0;
  if (p.temperature) temp = p.temperature[row];
  if (p.top_k) topk = p.top_k[row];
  if (p.top_p) topp = p.top_p[row];
  if (p.min_p) minp = p.min_p[row];
  int32_t ksel = p.k_max;
  if (kSel && p.k_sel) ksel = p.k_sel[row];
  if (kTopn) topk = p.k_max;
  uint64_t sd = 0ull, st = 0ull;
  uint32_t rid = (uint32_t)row;
  if (MODE & MODE_SAMPLE) {
    if (p.seed) sd = p.seed[row];
    if (p.step) st = p.step[row];
    if (p.row_id) rid = p.row_id[row];
  }

  // ---------------- wait for this row's slice ----------------
    bool timeout = dead;
    if (p.tma) {
      if (pending && !dead) {
        if (mbar_wait_bounded(&sh.bar[warp], (uint32_t)(uses & 1), p.wait_cycles)) {
          ++uses;
          pending = false;
          inflight = false;
        } else {
          timeout = true;   // the phase stays armed; no further copies are issued (the cluster is dead)
        }
      }
      // the (< 16 byte) tail of the slice, by its owner thread with plain loads
      const int64_t b16 = (cta_n * ES) & ~(int64_t)15;
      const int64_t tail_e0 = b16 / ES;
      if (!timeout && tail_e0 < cta_n && t == (int)(tail_e0 / ((int64_t)qr * VE))) {
        for (int64_t e = tail_e0; e < cta_n; ++e) {
          const int64_t se = slice_elem(e);
          if (ES == 4) reinterpret_cast<uint32_t*>(slice)[se] = reinterpret_cast<const uint32_t*>(grow)[e];
          else reinterpret_cast<uint16_t*>(slice)[se] = reinterpret_cast<const uint16_t*>(grow)[e];
        }
      }
    } else {
      for (int64_t e = 0; e < E.thr_n; ++e) {
        const int64_t le = (int64_t)t * qr * VE + e;
        const int64_t se = slice_elem(le);
        if (ES == 4) reinterpret_cast<uint32_t*>(slice)[se] = reinterpret_cast<const uint32_t*>(grow)[le];
        else reinterpret_cast<uint16_t*>(slice)[se] = reinterpret_cast<const uint16_t*>(grow)[le];
      }
    }
    __syncthreads();
    // This warp is done reading its region of the slice for this row: copy the cluster's next row
    // into it (first thing after the last pass over the row, so HBM streams while the row finishes).
    bool refilled = false;
    auto refill = [&]() {
      if (refilled) return;
      refilled = true;
      const int64_t nr = row + G;
      if (!p.tma || dead || nr >= p.B) return;
      __syncwarp();
      if (lane == 0) {
        fence_proxy_async_shared();
        inflight = issue_warp(nr);
      }
      pending = true;
    };

  // ---------------- P1: maximum (minimum for cut descriptors and radix searches), non-finite check --------
  constexpr bool kMin = (MODE & (MODE_CUT | MODE_SELECT | MODE_SAMPLE | MODE_TOPN | MODE_KEPT)) != 0;
  float mx = -INFINITY, mn = INFINITY, nf = 0.f;
  // the top-k select also counts the elements equal to the thread's running maximum (a select whose k lies
  // inside the row maximum's tie group then needs no radix search)
  float cmx = -INFINITY;
  uint32_t ccount = 0u;
  auto count_max = [&](float x) {
    const bool gt = x > cmx;
    ccount = gt ? 1u : ccount + (x == cmx ? 1u : 0u);
    cmx = gt ? x : cmx;
  };
  {
    const int nfull = E.thr_n / VE;
    if constexpr (VE == 8) {
      // bf16: packed maximum / minimum; x * 0 (or x != x for the top-k select) flags non-finite values
      const __nv_bfloat162 zero2 = __float2bfloat162_rn(0.f);
      __nv_bfloat162 mx2 = __float2bfloat162_rn(-INFINITY), mn2 = __float2bfloat162_rn(INFINITY), nf2 = zero2;
      for (int j = 0; j < nfull; ++j) {
        const uint4 v = E.mine[j];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const __nv_bfloat162 a = Tr::pair(w[h]);
          mx2 = __hmax2(mx2, a);
          if (kMin) mn2 = __hmin2(mn2, a);
          nf2 = kSel ? __hmax2(nf2, __hneu2(a, a)) : __hfma2(a, zero2, nf2);
        }
        if (kSel) {
          float x[VE];
          Tr::values(v, x);
#pragma unroll
          for (int i = 0; i < VE; ++i) count_max(x[i]);
        }
      }
      mx = fmaxf(__low2float(mx2), __high2float(mx2));
      mn = fminf(__low2float(mn2), __high2float(mn2));
      const float n0 = __low2float(nf2), n1 = __high2float(nf2);
      nf = (n0 != 0.f || n1 != 0.f) ? 1.f : 0.f;     // NaN compares unequal as well
    } else {
      for (int j = 0; j < nfull; ++j) {
        float x[VE];
        Tr::values(E.mine[j], x);
#pragma unroll
        for (int i = 0; i < VE; ++i) {
          mx = fmaxf(mx, x[i]);
          if (kMin) mn = fminf(mn, x[i]);
          // x * 0 is NaN for +-inf and NaN; the top-k select only rejects NaN
          nf = kSel ? (x[i] != x[i] ? 1.f : nf) : fmaf(x[i], 0.f, nf);
          if (kSel) count_max(x[i]);
        }
      }
    }
    const int tail = E.thr_n - nfull * VE;
    if (tail) {
      float x[VE];
      Tr::values(E.mine[nfull], x);
#pragma unroll
      for (int i = 0; i < VE; ++i) {
        if (i < tail) {
          mx = fmaxf(mx, x[i]);
          if (kMin) mn = fminf(mn, x[i]);
          nf = kSel ? (x[i] != x[i] ? 1.f : nf) : fmaf(x[i], 0.f, nf);
          if (kSel) count_max(x[i]);
        }
      }
    }
  }
  const float thr_mx = mx;   // this thread's maximum, before the reductions
  E.passes = 1;
  float M, Mmin;
  uint32_t gflags;
  uint32_t cMax = 0u;   // the top-k select: elements equal to the row maximum
  {
    const uint32_t bad = (nf != 0.f) ? 1u : 0u;    // NaN compares unequal as well
    mx = warp_max_f(mx);
    mn = -warp_max_f(-mn);
    const uint32_t flags = __reduce_or_sync(kFullMask, bad | (timeout ? 2u : 0u));
    const uint32_t wcount = kSel ? warp_sum_u32(cmx == mx ? ccount : 0u) : 0u;
    if (lane == 0) sh.ws[E.xc & 1][warp][0] = make_uint4(__float_as_uint(mx), __float_as_uint(mn), flags, wcount);
    E.exchange();
    // every warp reduces every warp's slot (no broadcast barrier)
    float m = -INFINITY, m2 = INFINITY;
    uint32_t fl = 0;
    for (int i = lane; i < C * Eng::NW; i += 32) {
      const uint4 v = E.wslot(i / Eng::NW, i % Eng::NW, 0);
      m = fmaxf(m, __uint_as_float(v.x));
      m2 = fminf(m2, __uint_as_float(v.y));
      fl |= v.z;
    }
    M = warp_max_f(m);
    Mmin = -warp_max_f(-m2);
    gflags = __reduce_or_sync(kFullMask, fl);
    if (kSel) {
      uint32_t c = 0u;
      for (int i = lane; i < C * Eng::NW; i += 32) {
        const uint4 v = E.wslot(i / Eng::NW, i % Eng::NW, 0);
        c += __uint_as_float(v.x) == M ? v.w : 0u;
      }
      cMax = warp_sum_u32(c);
    }
    E.exchange_done();
  }
  if (gflags & 2u) dead = true;

  // ---------------- row status and parameters (uniform over the cluster) ----------------
  int status = VSAMP_OK;
  if (bad_len) status = VSAMP_ERR_INVALID_ARG;
  else if (gflags & 2u) status = VSAMP_ERR_TIMEOUT;
  else if (gflags & 1u) status = VSAMP_ERR_NONFINITE;
  else if (kSel && ksel > p.k_max) status = VSAMP_ERR_INVALID_ARG;
  else if (kCutLike && (isnan(temp) || isinf(temp) || isnan(topp) || !(topp > 0.f) || isnan(minp) || minp > 1.f))
    status = VSAMP_ERR_INVALID_ARG;
  else if ((MODE & (MODE_LSE | MODE_LOGPROB)) && (isnan(temp) || isinf(temp)))
    status = VSAMP_ERR_INVALID_ARG;
  int32_t tok_in = 0;
  if ((MODE & (MODE_LOGPROB | MODE_KEPT)) && status == VSAMP_OK) {
    tok_in = p.token_in[row];
    if (tok_in < 0 || (int64_t)tok_in >= n) status = VSAMP_ERR_INVALID_ARG;
  }
  // T <= 0 means greedy sampling; a top-N list is the same at every temperature (T <= 0 read as 1)
  const bool greedy = !kTopn && !(temp > 0.f);
  const float Teff = temp > 0.f ? temp : 1.f;
  const float invT = 1.f / Teff;
  const float c1 = kLog2e * invT;
  bool minp_on = kCutLike && !greedy && minp > 0.f;
  const unsigned long long one = 1ull << kMassShift;     // fixed-point mass of a maximum token

  // min-p keeps w >= minp  <=>  x >= x* = M + T ln(minp). x* is formed as an unevaluated sum hi + lo
  // (exact product and sum corrections), and the threshold is the smallest fp32 value >= x*.
  if (minp_on && status == VSAMP_OK) {
    const float L = logf(minp);
    const float ph = Teff * L, pl = fmaf(Teff, L, -ph);        // T*L = ph + pl exactly
    const float sh_ = M + ph;                                   // M + ph = sh_ + sl exactly
    const float bb = sh_ - M;
    const float sl = (M - (sh_ - bb)) + (ph - bb);
    const float lo = sl + pl;
    const float xf = lo > 0.f ? nextafterf(sh_, INFINITY) : sh_;
    plan.kmin32 = key_f32_bits(__float_as_uint(xf));
    // a threshold at or below the row's minimum keeps every token: the filter is off
    if (plan.kmin32 <= key_f32_bits(__float_as_uint(Mmin))) minp_on = false;
  }

  unsigned long long Sfx = 0, cM = 0;
  uint32_t cm_thr = 0, cm_pre = 0;   // this thread's maxima, and the maxima before its chunk (index order)
  float xP = -INFINITY;          // kept: x > xP, or x == xP and index <= It
  int32_t It = kAllIndex;
  int32_t boundary = kNoIndex;   // global index of the last kept token, if this thread holds it
  bool fin_valid = false;
  Cut fin{};

  if (status == VSAMP_OK) {
    if (!kSel) {
      // ---------------- P2: fixed-point sum, maxima per thread, min-p statistics ----------------
      const MassPart mp = minp_on ? mass_pass<T, true>(E.mine, E.thr_n, M, c1, plan.kmin32)
                                  : mass_pass<T, false>(E.mine, E.thr_n, M, c1, 0u);
      unsigned long long s_loc = mp.s, mge = mp.mge;
      uint32_t cm_loc = mp.cm, cge = mp.cge, minkey = mp.minkey, cmin = mp.cmin;
      E.passes += 1;
      uint32_t cm_incl = cm_loc;      // inclusive prefix of the maxima counts within the warp
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const uint32_t y = __shfl_up_sync(kFullMask, cm_incl, o);
        if (lane >= o) cm_incl += y;
      }
      cm_thr = cm_loc;
      s_loc = warp_sum_u64(s_loc);
      cm_loc = __shfl_sync(kFullMask, cm_incl, 31);
      if (minp_on) {
        mge = warp_sum_u64(mge);
        cge = warp_sum_u32(cge);
        const uint32_t mk = warp_min_u32(minkey);
        cmin = warp_sum_u32(minkey == mk ? cmin : 0u);
        minkey = mk;
      }
      if (lane == 0) {
        uint4* ws = sh.ws[E.xc & 1][warp];
        ws[0] = make_uint4((uint32_t)s_loc, (uint32_t)(s_loc >> 32), cm_loc, cge);
        ws[1] = make_uint4((uint32_t)mge, (uint32_t)(mge >> 32), minkey, cmin);
      }
      E.exchange();
      // every warp reduces every warp's slot (no broadcast barrier); the slots are in index order
      // (CTA rank, then warp), so the maxima of the slots before this warp's give its prefix
      unsigned long long mass_ge = 0ull;
      uint32_t cnt_ge = 0, minkey_ge = 0xFFFFFFFFu, cnt_minkey = 0;
      {
        const int mine_slot = crank * Eng::NW + warp;
        unsigned long long a = 0, b = 0;
        uint32_t c = 0, cb = 0, d = 0, mk = 0xFFFFFFFFu, cc = 0;
        for (int i = lane; i < C * Eng::NW; i += 32) {
          const uint4 v0 = E.wslot(i / Eng::NW, i % Eng::NW, 0);
          a += ((unsigned long long)v0.y << 32) | v0.x;
          c += v0.z;
          if (i < mine_slot) cb += v0.z;
          if (minp_on) {
            const uint4 v1 = E.wslot(i / Eng::NW, i % Eng::NW, 1);
            d += v0.w;
            b += ((unsigned long long)v1.y << 32) | v1.x;
            if (v1.z < mk) { mk = v1.z; cc = v1.w; }
            else if (v1.z == mk) cc += v1.w;
          }
        }
        Sfx = warp_sum_u64(a);
        cM = warp_sum_u32(c);
        cm_pre = warp_sum_u32(cb) + (cm_incl - cm_thr);   // maxima before this thread's chunk
        if (minp_on) {
          mass_ge = warp_sum_u64(b);
          cnt_ge = warp_sum_u32(d);
          minkey_ge = warp_min_u32(mk);
          cnt_minkey = warp_sum_u32(mk == minkey_ge ? cc : 0u);
        }
      }
      E.exchange_done();
      // ---------------- per-row plan ----------------
      {
        plan.status = VSAMP_OK;
        plan.path = p.tma ? 0 : PATH_NOTMA;
        plan.logS = logf(u64_to_float(Sfx) * 9.094947017729282379e-13f);   // 2^-40
        plan.ck_mode = 0;
        plan.cp_mode = 0;
        plan.goal_p = -1.f;
        plan.cp_goal = 0;
        if (kCutLike) {
          const uint32_t rkM = Tr::rkey_of_value(M);
          if (greedy) {
            plan.fin = Cut{rkM, 0, 1, cM, one, 0};
            plan.path |= PATH_MAXGROUP;
          } else {
            const bool topk_on = topk > 0 && (int64_t)topk < n;
            const bool topp_on = topp < 1.f;
            const unsigned long long keff = topk_on ? (unsigned long long)topk : (unsigned long long)n;
            if (topk_on) {
              if (keff <= cM) {
                plan.ck = Cut{rkM, 0, keff, cM, keff * one, 0};
                plan.ck_mode = 1;
              } else {
                plan.ck = Cut{0, 0, keff, 0, 0, 0};
                plan.ck_mode = 2;
              }
            }
            if (topp_on) {
              if (plan.ck_mode != 2) {
                const unsigned long long Sk = topk_on ? plan.ck.mass : Sfx;
                const unsigned long long target = ceil_mul_frac(topp, Sk);
                if (target <= cM * one) {
                  unsigned long long need = (target + one - 1) >> kMassShift;
                  need = need < 1 ? 1 : need;
                  plan.cp = Cut{rkM, 0, need, cM, need * one, 0};
                  plan.cp_mode = 1;
                } else {
                  plan.cp_mode = 2;
                  if (topk_on) plan.cp_goal = target;
                  else plan.goal_p = topp;
                }
              } else if (ceil_mul_frac(topp, Sfx) <= one) {
                // target <= p * S <= one maximum's mass: the first maximum alone reaches it
                plan.cp = Cut{rkM, 0, 1, cM, one, 0};
                plan.cp_mode = 1;
              } else {
                plan.cp_mode = 2;   // goal from the top-k mass, after the top-k rounds
              }
            }
            // top-p keeping the first maximum alone is the shortest cut: no radix search for top-k
            if (plan.cp_mode == 1 && plan.cp.kept() == 1 && plan.ck_mode == 2) plan.ck_mode = 0;
            if (plan.ck_mode == 1 || plan.cp_mode == 1) plan.path |= PATH_MAXGROUP;
            if (minp_on) {
              // min-p keeps the whole group of the smallest key at or above its threshold
              const uint32_t rkm = (Tr::KB == 32) ? minkey_ge : (minkey_ge >> 16);
              plan.fin = Cut{rkm, (unsigned long long)(cnt_ge - cnt_minkey), cnt_minkey, cnt_minkey, mass_ge, 1};
            } else {
              // no filter binds: every token. The prefix ends with the row minimum's group; only the cut
              // descriptor needs that group (a one-token row's minimum is its maximum).
              const uint32_t rk_last = (MODE & MODE_CUT) ? Tr::rkey_of_value(Mmin) : rkM;
              plan.fin = Cut{rk_last, 0, (unsigned long long)n, 0, Sfx, 1};
            }
          }
        }
      }
      if (kCutLike && !greedy) {
        // ---------------- radix rounds where the cut leaves the maximum's group ----------------
        if (plan.ck_mode == 2) {
          // a count search; the kept mass, where the top-p goal needs it, in one pass after it
          const RadixOut r = E.radix_search(false, plan.ck.need, -1.f, false, M, c1, 0u, Mmin);
          {
            if (!r.ok) plan.status = VSAMP_ERR_INVALID_ARG;
            const unsigned long long need = plan.ck.need - r.cnt_above;
            const unsigned long long wP = mass_fx(ex2_approx((Tr::value_of_rkey(r.rk) - M) * c1));
            const bool want_mass = plan.cp_mode == 2 || (MODE & MODE_KEPT) != 0;
            const unsigned long long above = want_mass ? E.mass_above_key(r.rk, M, c1, r.vsel) : 0ull;
            plan.ck = Cut{r.rk, r.cnt_above, need, r.cnt_eq, above + need * wP, 0};
            plan.path |= PATH_RADIX_K;
            if (plan.cp_mode == 2) plan.cp_goal = ceil_mul_frac(topp, plan.ck.mass);
          }
        }
        if (plan.cp_mode == 2 && plan.status == VSAMP_OK) {
          // after a top-k cut the goal lies within the keys at or above its pivot
          const uint32_t floor_rk = plan.ck_mode == 2 ? plan.ck.rk : 0u;
          const RadixOut r = E.radix_search(true, plan.cp_goal, plan.goal_p, true, M, c1, floor_rk, Mmin);
          {
            if (!r.ok) plan.status = VSAMP_ERR_INVALID_ARG;
            const unsigned long long wP = mass_fx(ex2_approx((Tr::value_of_rkey(r.rk) - M) * c1));
            // a group element is kept while the mass before it is below the target
            unsigned long long need = wP ? (r.goal + wP - 1) / wP : 1;
            need = need < 1 ? 1 : (need > r.cnt_eq ? r.cnt_eq : need);
            plan.cp = Cut{r.rk, r.cnt_above, need, r.cnt_eq, r.mass_above + need * wP, 0};
            plan.path |= PATH_RADIX_P;
          }
        }
        // ---------------- the shortest prefix wins ----------------
        {
          Cut best = plan.fin;   // the min-p cut, or every token
          if (plan.ck_mode && plan.ck.kept() < best.kept()) best = plan.ck;
          if (plan.cp_mode && plan.cp.kept() < best.kept()) best = plan.cp;
          if (minp_on && best.whole) plan.path |= PATH_MINP;
          plan.fin = best;
        }
      }
      status = plan.status;
      fin = plan.fin;
      fin_valid = kCutLike && status == VSAMP_OK;
    } else {
      // ---------------- stand-alone top-k select ----------------
      if (ksel <= 0) {
        fin = Cut{0u, 0, 0, 0, 0, 0};
      } else if (ksel >= n) {
        fin = Cut{0u, 0, (unsigned long long)n, 0, 0, 1};
      } else if ((int64_t)cMax >= (int64_t)ksel) {
        // k inside the maximum's tie group: the first k maxima by index, no radix search
        fin = Cut{Tr::rkey_of_value(M), 0, (unsigned long long)ksel, cMax, 0, 0};
      } else {
        const RadixOut r = E.radix_search(false, (unsigned long long)ksel, -1.f, false, M, c1, 0u, Mmin);
        if (!r.ok) status = VSAMP_ERR_INVALID_ARG;
        fin = Cut{r.rk, r.cnt_above, (unsigned long long)ksel - r.cnt_above, r.cnt_eq, 0, 0};
      }
      fin_valid = status == VSAMP_OK;
    }
  }

  // ---------------- the cut's last kept index, per thread ----------------
  bool select_none = false;
  if (fin_valid) {
    const bool need_boundary = !fin.whole || (MODE & MODE_CUT) || ((MODE & MODE_SAMPLE) && fin.kept() == 1);
    if (kSel && fin.need == 0 && fin.above == 0) {
      select_none = true;
      xP = INFINITY;
      It = kNoIndex;
    } else if (!need_boundary) {
      // every element of the group is kept and no output needs the boundary index
      const bool every_token = fin.above == 0 && fin.cnt_eq == 0;
      xP = every_token ? -INFINITY : Tr::value_of_rkey(fin.rk);
      It = kAllIndex;
    } else {
      xP = Tr::value_of_rkey(fin.rk);
      unsigned long long need = fin.need, start, cnt;
      if (!kSel && fin.rk == Tr::rkey_of_value(M)) {
        // the group of maxima: P2 counted them per thread and prefixed them over the cluster
        start = cm_pre;
        cnt = cm_thr;
        if (fin.whole) need = cM;
      } else {
        E.count_equal_pass(xP);
        const uint32_t ctot = E.block_scan_tcount();
        uint32_t cpre, total;
        E.cluster_prefix_u32(ctot, 0, cpre, total);
        start = (unsigned long long)cpre + sh.tpre[t];
        cnt = sh.tcount[t];
        if (fin.whole) need = total;     // the last element of the group
      }
      It = E.local_cut_index(xP, need, start, cnt, boundary);
    }
  }

  // ---------------- P4: Gumbel-max draw over the kept prefix ----------------
  int32_t out_token = -1;
  float out_s = 0.f;         // (x - M) / T of the drawn token
  bool last_cta = false;     // this warp reduced the row's arg-max and writes the draw's outputs
  if ((MODE & MODE_SAMPLE) && fin_valid) {
    const unsigned long long kept = fin.kept();
    if (greedy || kept == 1) {
      // the first maximum: written by the thread that holds it
      if (boundary >= 0) {
        p.token[row] = boundary;                                  // a maximum: (x - M) / T = 0
        if (p.logprob) p.logprob[row] = fminf(-plan.logS, 0.f);
      }
    } else {
      {
        // prune bound: a token can beat B0 = ln(S_kept) - 3 only if u < w * kappa, kappa = e^3 / S_kept
        const float skept = fmaxf(u64_to_float(fin.mass) * 9.094947017729282379e-13f, 1.f);   // 2^-40
        const float kappa = 20.085536923187668f / skept;
        plan.kappa = kappa;
        plan.all_cand = kappa >= 0.99f;
        plan.bk = plan.all_cand ? 0xFFFFFFFFu : __float2uint_ru(kappa * 1.00001f * 4294967296.0f);
        plan.b0 = -logf(kappa);
      }
      const PhiloxKey key{(uint32_t)sd, (uint32_t)(sd >> 32)};
      const uint32_t st_lo = (uint32_t)st, st_hi = (uint32_t)(st >> 32);
      const float kappa = plan.kappa;
      const uint32_t bk = plan.bk;
      const float B0 = plan.b0;
      {
        const bool all_cand = plan.all_cand;
        const int nfull = E.thr_n / VE;
        // leading full vectors whose tokens equal to the pivot value are all kept: e0 + VE - 1 <= It
        int jfull = 0;
        {
          const int64_t lim = (int64_t)It - E.thr_e0 - (VE - 1);
          if (lim >= 0) jfull = (int)(lim / VE + 1 < (int64_t)nfull ? lim / VE + 1 : (int64_t)nfull);
        }
        const uint32_t g0 = (uint32_t)(E.thr_e0 >> 2);      // Philox counter of the thread's first 4 tokens
        // Main pass: a vector is flagged when one of its kept tokens' words is below the prune bound bk
        // (about e^3 tokens per row); flagged vectors are evaluated exactly below. When every kept token
        // is a candidate, every vector holding a kept token is flagged.
        unsigned long long flagged =
            all_cand ? kept_vectors<T>(E.mine, E.thr_n, E.thr_e0, xP, It)
                     : draw_pass<T>(E.mine, E.thr_n, E.thr_e0, jfull, xP, It, g0, rid, st_lo, st_hi, key, bk);
        // Flagged vectors: the kept tokens whose word passes the bound get the exact perturbed score.
        float bscore = -INFINITY, bs = 0.f;
        int32_t bidx = 0x7FFFFFFF;
        while (flagged) {
          const int j = __ffsll((long long)flagged) - 1;
          flagged &= flagged - 1ull;
          const uint4 v = E.mine[j];
          float x[VE];
          Tr::values(v, x);
          const int cnt = j < nfull ? VE : E.thr_n - nfull * VE;
          const int64_t e0 = E.thr_e0 + (int64_t)j * VE;
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
        E.passes += 1;
        refill();    // this warp has finished reading its region of the slice
        // ---------------- lock-free cluster arg-max ----------------
        // Two levels, no barrier: each warp publishes its partial and counts itself in with an
        // acquire-release atomic; the last warp of each CTA reduces its CTA's partials and publishes them
        // in CTA 0; the last of those reduces the cluster's and writes the row's outputs. Every other warp
        // goes straight on to its next row.
        const ArgMax best = warp_argmax(ArgMax{bscore, bidx, bs});
        int32_t wcut = boundary;  // the cut's boundary index, if this warp holds it (else -1)
#pragma unroll
        for (int o = 16; o; o >>= 1) wcut = max(wcut, __shfl_xor_sync(kFullMask, wcut, o));
        const int par = (int)(k & 1);
        // level 1: each warp publishes its partial in its CTA and counts itself in; the CTA's last warp
        // reduces the CTA's partials
        uint32_t old = 0;
        if (lane == 0) {
          sh.apart[par][warp] = make_uint4(__float_as_uint(best.score), (uint32_t)best.idx, __float_as_uint(best.s),
                                           (uint32_t)wcut);
          old = smem_atomic_add_acq_rel_cta(&sh.lcnt[par], 1u);
        }
        old = __shfl_sync(kFullMask, old, 0);
        if (old == (uint32_t)(Eng::NW - 1)) {
          __syncwarp();
          ArgMax c2{-INFINITY, 0x7FFFFFFF, 0.f};
          int32_t ccut = -1;
          if (lane < Eng::NW) {
            const uint4 v = sh.apart[par][lane];
            c2 = ArgMax{__uint_as_float(v.x), (int32_t)v.y, __uint_as_float(v.z)};
            ccut = (int32_t)v.w;
          }
          c2 = warp_argmax(c2);
#pragma unroll
          for (int o = 16; o; o >>= 1) ccut = max(ccut, __shfl_xor_sync(kFullMask, ccut, o));
          // level 2: the CTA's partial goes to CTA 0; the cluster's last warp reduces the C partials
          uint32_t old2 = 0;
          if (lane == 0) {
            sh.lcnt[par] = 0u;
            if (C > 1) {
              dsmem_store_v4(dsmem_map(&sh.aslot[par][crank], 0), __float_as_uint(c2.score), (uint32_t)c2.idx,
                             __float_as_uint(c2.s), (uint32_t)ccut);
              old2 = dsmem_atomic_add_acq_rel(dsmem_map(&sh.acnt[par], 0), 1u);
            }
          }
          old2 = __shfl_sync(kFullMask, old2, 0);
          if (C == 1 || old2 == (uint32_t)(C - 1)) {
            __syncwarp();
            last_cta = true;        // this warp writes the row's outputs
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
            const bool certified = all_cand || (g.score > B0 + 1e-4f * fmaxf(1.f, fabsf(B0)));
            if (certified) {
              out_token = g.idx;
              out_s = g.s;
            } else {
              // the prune bound did not certify the draw (probability ~1e-9): this warp evaluates every
              // kept token of the row from global memory
              plan.path |= PATH_FALLBACK;
              const int32_t Ig = cut < 0 ? kAllIndex : cut;
              float fs = -INFINITY, fsv = 0.f;
              int32_t fi = 0x7FFFFFFF;
              for (int64_t e = lane; e < n; e += 32) {
                const float xv = Tr::load_global(p.x, (int64_t)row * p.ld + e);
                if (!(xv > xP || (xv == xP && e <= (int64_t)Ig))) continue;
                const uint4 w4 = philox4x32_10(make_uint4((uint32_t)(e >> 2), rid, st_lo, st_hi), key);
                const uint32_t bw = philox_word(w4, (int)(e & 3));
                const float sv = (xv - M) * invT;
                const float score = gumbel_score(sv, bw);
                if (argmax_better(score, (int32_t)e, fs, fi)) { fs = score; fi = (int32_t)e; fsv = sv; }
              }
              const ArgMax fb = warp_argmax(ArgMax{fs, fi, fsv});
              out_token = fb.idx;
              out_s = fb.s;
            }
          }
        }
      }
    }
  }

  // ---------------- top-k select / top-N emission (ascending index order) ----------------
  if (kSel || kTopn) {
    int32_t* orow = p.out_idx + (int64_t)row * p.k_max;
    uint32_t total = 0;
    if (fin_valid && !select_none) {
      // a thread whose maximum is below the cut, or equal to it with the boundary before its chunk, keeps nothing
      const bool none_here = !(thr_mx > xP || (thr_mx == xP && (int64_t)It >= E.thr_e0));
      uint32_t c = 0;
      if (!none_here)
        E.for_each([&](int64_t e, float x) { c += (x > xP || (x == xP && e <= (int64_t)It)) ? 1u : 0u; });
      sh.tcount[t] = c;
      const uint32_t ctot = E.block_scan_tcount();
      uint32_t cpre;
      E.cluster_prefix_u32(ctot, 1, cpre, total);
      uint32_t pos = cpre + sh.tpre[t];
      if (c)
        E.for_each([&](int64_t e, float x) {
          if (x > xP || (x == xP && e <= (int64_t)It)) {
            if (pos < (uint32_t)p.k_max) orow[pos] = (int32_t)e;
            ++pos;
          }
        });
      E.passes += 2;
    }
    if (crank == 0)
      for (int64_t j = (int64_t)total + t; j < p.k_max; j += NT) orow[j] = -1;
  }

  // ---------------- mask ----------------
  if (MODE & MODE_MASK) {
    // one VE-byte store per vector (8 bytes for bf16, 4 for fp32) where the mask row allows it
    uint8_t* mrow = p.mask + (int64_t)row * p.V;
    const bool vec_ok = ((reinterpret_cast<uintptr_t>(mrow) + (uintptr_t)E.thr_e0) & (uintptr_t)(VE - 1)) == 0;
    const int nvec = (E.thr_n + VE - 1) / VE;
    for (int j = 0; j < nvec; ++j) {
      float x[VE];
      Tr::values(E.mine[j], x);
      const int64_t e0 = E.thr_e0 + (int64_t)j * VE;
      const int cnt = E.thr_n - j * VE < VE ? E.thr_n - j * VE : VE;
      uint32_t b[2] = {0u, 0u};
#pragma unroll
      for (int i = 0; i < VE; ++i) {
        const bool k = fin_valid && i < cnt && (x[i] > xP || (x[i] == xP && e0 + i <= (int64_t)It));
        b[i >> 2] |= (k ? 1u : 0u) << (8 * (i & 3));
      }
      if (vec_ok && cnt == VE) {
        if (VE == 8) *reinterpret_cast<uint2*>(mrow + e0) = make_uint2(b[0], b[1]);
        else *reinterpret_cast<uint32_t*>(mrow + e0) = b[0];
      } else {
        for (int i = 0; i < cnt; ++i) mrow[e0 + i] = (uint8_t)((b[i >> 2] >> (8 * (i & 3))) & 1u);
      }
    }
  }

  // ---------------- finalisation ----------------
  if ((MODE & MODE_CUT) && fin_valid && boundary >= 0) p.cut[row].idx_cut = boundary;
  // the kept-set log-probability: written by the thread whose chunk holds the token (its cut index It
  // decides whether the token is kept)
  if ((MODE & MODE_KEPT) && fin_valid && (int64_t)tok_in >= E.thr_e0 && (int64_t)tok_in < E.thr_e0 + E.thr_n) {
    const float xt = Tr::load_global(p.x, (int64_t)row * p.ld + tok_in);
    const bool kept = xt > xP || (xt == xP && tok_in <= It);
    const float log_sk = logf(u64_to_float(fin.mass) * 9.094947017729282379e-13f);   // 2^-40
    p.logprob[row] = kept ? fminf((xt - M) * invT - log_sk, 0.f) : -INFINITY;
  }
  // the row's outputs come from thread 0, except a Gumbel draw's, which come from lane 0 of the warp
  // that reduced it
  const bool p4_path = (MODE & MODE_SAMPLE) && fin_valid && !(greedy || fin.kept() == 1);
  const bool writer = p4_path ? last_cta : (crank == 0 && warp == 0);
  if (writer && lane == 0) {
    if (MODE & MODE_LSE) {
      if (p.row_max) p.row_max[row] = status == VSAMP_OK ? M : __int_as_float(0x7FC00000);
      if (p.row_logsum) p.row_logsum[row] = status == VSAMP_OK ? (float)plan.logS : __int_as_float(0x7FC00000);
    }
    if ((MODE & MODE_KEPT) && !fin_valid) p.logprob[row] = __int_as_float(0x7FC00000);
    if (MODE & MODE_LOGPROB) {
      float lp = __int_as_float(0x7FC00000);
      if (status == VSAMP_OK) {
        const float xt = Tr::load_global(p.x, (int64_t)row * p.ld + tok_in);
        lp = fminf((xt - M) * invT - plan.logS, 0.f);
      }
      if (p.logprob) p.logprob[row] = lp;
    }
    if (MODE & MODE_SAMPLE) {
      const bool one_token = fin_valid && (greedy || fin.kept() == 1);
      if (!fin_valid) {
        p.token[row] = -1;
        if (p.logprob) p.logprob[row] = __int_as_float(0x7FC00000);
      } else if (!one_token) {
        if (out_token >= 0 && (int64_t)out_token < n) {
          p.token[row] = out_token;
          if (p.logprob) p.logprob[row] = fminf(out_s - plan.logS, 0.f);
        } else {
          status = VSAMP_ERR_INVALID_ARG;
          p.token[row] = -1;
          if (p.logprob) p.logprob[row] = __int_as_float(0x7FC00000);
        }
      }
    }
    if (MODE & MODE_CUT) {
      vsamp_cut& c = p.cut[row];
      c.status = status;
      if (fin_valid) {
        c.pivot_key = Tr::key32(fin.rk);
        c.kept = (int32_t)fin.kept();
      } else {
        c.pivot_key = 0;
        c.idx_cut = -1;
        c.kept = 0;
      }
    }
    if (p.row_status) p.row_status[row] = status;
    if (p.stats) {
      p.stats[row * 4 + 0] = E.passes;
      p.stats[row * 4 + 1] = E.rounds;
      p.stats[row * 4 + 2] = fin_valid ? (int32_t)fin.kept() : 0;
      p.stats[row * 4 + 3] = (kSel || !fin_valid) ? (p.tma ? 0 : PATH_NOTMA) : plan.path;
    }
  }
    refill();
    __syncthreads();
  }
  // after a timed-out load, wait (again bounded, ~2 s) for a bulk copy of this warp that may still be
  // landing in shared memory before the CTA leaves
  if (p.tma && inflight) (void)mbar_wait_bounded(&sh.bar[warp], (uint32_t)(uses & 1), 4000000000LL);
  // no CTA may leave while a peer can still read its shared memory
  E.cluster.sync();
  (void)q;
}

}  // namespace vsamp
