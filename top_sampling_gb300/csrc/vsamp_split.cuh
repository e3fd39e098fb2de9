// The split-vocabulary sampling path (vsamp_sample_ws, vsamp_sample_static): every row is cut into fixed pieces of
// 4 KB (2048 bf16 or 1024 fp32 logits) and one fused streaming kernel sweeps all (row, piece) pairs of the batch
// (see "The fused streaming sampler" below). The cut into pieces depends only on V, so results are deterministic
// and do not depend on the batch.
#pragma once

#include "vsamp_row.cuh"

namespace vsamp {

constexpr int kSplitThreads = 256;
constexpr int kStreamThreads = 256;  // threads per CTA of the streaming kernels (independent warps)
constexpr int kPieceBytes = 4096;    // bytes of logits per piece (the unit of a warp's work and of the row statistics)
template <typename T>
constexpr int kPieceElems = kPieceBytes / Traits<T>::ESIZE;     // 2048 bf16 or 1024 fp32 logits
template <typename T>
constexpr int kPieceVecs = kPieceBytes / 32 / 16;               // 16-byte vectors per lane per piece: 8
constexpr int kDrawRun = 4;          // pieces of one row per draw item

struct ChunkStat {                   // 16 bytes per (row, chunk)
  float m;                           // chunk maximum (NaN flags a non-finite value)
  uint32_t cnt;                      // elements equal to m
  unsigned long long s;              // sum of 2^((x - m) * c1), 2^-40 fixed point
};

static_assert(sizeof(ChunkStat) == 16, "ChunkStat layout");

__host__ __device__ inline int64_t split_chunk_elems(int esize) { return kPieceBytes / esize; }
__host__ __device__ inline int64_t split_nchunks(int64_t V, int esize) {
  const int64_t k = split_chunk_elems(esize);
  return (V + k - 1) / k;
}

// orderable 32-bit key of a non-NaN float (larger float, larger key)
__device__ __forceinline__ uint32_t score_key(float s) {
  const uint32_t f = __float_as_uint(s);
  return (f & 0x80000000u) ? ~f : (f | 0x80000000u);
}
__device__ __forceinline__ float score_of_key(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// One 16-byte vector of a row: elements e .. e + VE - 1 (fewer past the row end); returns how many are
// valid. Aligned rows take one 16-byte load (LAST_USE: marked evict-first, for the draw's re-read; else the
// default policy keeps the chunk in L2 for it), others element loads.
template <typename T, bool LAST_USE>
__device__ __forceinline__ int load_vec(const Params& p, const unsigned char* xr, int64_t e, uint4& v) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  const int64_t left = p.V - e;
  const int cnt = left <= 0 ? 0 : (left >= VE ? VE : (int)left);
  if (cnt == VE && p.tma) {
    const uint4* src = reinterpret_cast<const uint4*>(xr + e * Tr::ESIZE);
    v = LAST_USE ? __ldcs(src) : *src;
  } else {
    uint32_t w[4] = {0u, 0u, 0u, 0u};
    for (int i = 0; i < cnt; ++i) {
      if (Tr::ESIZE == 4) w[i] = reinterpret_cast<const uint32_t*>(xr)[e + i];
      else w[i >> 1] |= (uint32_t)reinterpret_cast<const uint16_t*>(xr)[e + i] << (16 * (i & 1));
    }
    v = make_uint4(w[0], w[1], w[2], w[3]);
  }
  return cnt;
}

// A chunk statistic written by another CTA of the same launch: read through L2 (L1 is not coherent).
__device__ __forceinline__ ChunkStat load_stat(const ChunkStat* a) {
  const uint4 v = __ldcg(reinterpret_cast<const uint4*>(a));
  ChunkStat cs;
  cs.m = __uint_as_float(v.x);
  cs.cnt = v.y;
  cs.s = ((unsigned long long)v.w << 32) | v.z;
  return cs;
}

// ------------------------------------------------------------------------------------------------
// Block helpers (256 threads).
// ------------------------------------------------------------------------------------------------
struct SplitShared {
  float f[8];
  uint32_t u[8][4];
  unsigned long long q[8][2];
  int32_t i[8];
  uint32_t ticket;
  uint32_t bsel;
  unsigned long long bq[4];
  uint32_t hcnt[256];
  uint32_t hlo[256];
  uint32_t hhi[256];
};

__device__ __forceinline__ float block_max_f(float v, SplitShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_max_f(v);
  __syncthreads();
  if (lane == 0) sh.f[warp] = v;
  __syncthreads();
  float m = sh.f[0];
#pragma unroll
  for (int w = 1; w < kSplitThreads / 32; ++w) m = fmaxf(m, sh.f[w]);
  return m;
}
__device__ __forceinline__ unsigned long long block_sum_u64(unsigned long long v, SplitShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_u64(v);
  __syncthreads();
  if (lane == 0) sh.q[warp][0] = v;
  __syncthreads();
  unsigned long long s = 0;
#pragma unroll
  for (int w = 0; w < kSplitThreads / 32; ++w) s += sh.q[w][0];
  return s;
}
__device__ __forceinline__ uint32_t block_sum_u32(uint32_t v, SplitShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_sum_u32(v);
  __syncthreads();
  if (lane == 0) sh.u[warp][0] = v;
  __syncthreads();
  uint32_t s = 0;
#pragma unroll
  for (int w = 0; w < kSplitThreads / 32; ++w) s += sh.u[w][0];
  return s;
}
__device__ __forceinline__ uint32_t block_min_u32(uint32_t v, SplitShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  v = warp_min_u32(v);
  __syncthreads();
  if (lane == 0) sh.u[warp][1] = v;
  __syncthreads();
  uint32_t s = 0xFFFFFFFFu;
#pragma unroll
  for (int w = 0; w < kSplitThreads / 32; ++w) s = min(s, sh.u[w][1]);
  return s;
}
// exclusive prefix of v over threads in index order, and the block total
__device__ __forceinline__ uint32_t block_scan_u32(uint32_t v, uint32_t& total, SplitShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const uint32_t y = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += y;
  }
  __syncthreads();
  if (lane == 31) sh.u[warp][2] = incl;
  __syncthreads();
  uint32_t base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kSplitThreads / 32; ++w) {
    const uint32_t x = sh.u[w][2];
    if (w < warp) base += x;
    tot += x;
  }
  total = tot;
  return base + incl - v;
}

// ------------------------------------------------------------------------------------------------
// The row planner: the CTA whose chunk completes the row in stream_stats_kernel.
// ------------------------------------------------------------------------------------------------
template <typename T>
struct RowPlanner {
  using Tr = Traits<T>;
  static constexpr int VE = Tr::VE;
  const Params& p;
  SplitShared& sh;
  int64_t row, n;
  float M, c1;
  int passes = 0, rounds = 0;
  float Mmin = -INFINITY;   // the row's minimum (-inf when unknown: the first round then takes key bytes)

  // visits every element of the row in tiles of 256 vectors: f(index, value, valid); tile order is index order
  template <typename F>
  __device__ __forceinline__ void for_each_tile(int64_t begin_vec, F&& f) {
    const unsigned char* xr = p.x + (int64_t)row * p.ld * Tr::ESIZE;
    const int64_t nvec = (n + VE - 1) / VE;
    for (int64_t v0 = begin_vec; v0 < nvec; v0 += kSplitThreads) {
      const int64_t vi = v0 + threadIdx.x;
      float x[VE];
      int cnt = 0;
      if (vi < nvec) {
        const int64_t e = vi * VE;
        cnt = n - e >= VE ? VE : (int)(n - e);
        if (cnt == VE && p.tma) {
          Tr::values(reinterpret_cast<const uint4*>(xr)[vi], x);
        } else {
#pragma unroll
          for (int i = 0; i < VE; ++i) x[i] = i < cnt ? Tr::load_global(xr, e + i) : -INFINITY;
        }
      } else {
#pragma unroll
        for (int i = 0; i < VE; ++i) x[i] = -INFINITY;
      }
      if (!f(v0, vi * VE, x, cnt)) break;
    }
  }

  // radix search over the whole row (as the row engine's, with the row read from L2 by this CTA): a first
  // round of value bins over [Mmin, M] when that range is finite, then key rounds inside the selected bin
  __device__ __noinline__ RadixOut radix(bool mass_mode, unsigned long long goal, float goal_p, bool want_mass) {
    RadixOut out{};
    out.ok = 1;
    uint32_t prefix = 0;
    unsigned long long cnt_above = 0, mass_above = 0;
    const bool hist_mass = want_mass || mass_mode;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    const ValueBins vb = make_value_bins(Mmin, M);
    bool vround = vb.sc > 0.f, first = true;
    uint32_t klo = 0u, khi = 0xFFFFFFFFu;
    int shift = vround ? 0 : Tr::KB - 8;
    for (;;) {
      __syncthreads();
      for (int b = t; b < 256; b += kSplitThreads) { sh.hcnt[b] = 0; sh.hlo[b] = 0; sh.hhi[b] = 0; }
      __syncthreads();
      const int hi_shift = shift + 8;
      const uint32_t hmask = hi_shift >= 32 ? 0u : (0xFFFFFFFFu << hi_shift);
      for_each_tile(0, [&](int64_t, int64_t, const float (&x)[VE], int cnt) {
        uint32_t run_bin = 0xFFFFFFFFu, run_cnt = 0;
        unsigned long long run_mass = 0;
        auto flush = [&]() {
          if (run_cnt) {
            atomicAdd(&sh.hcnt[run_bin], run_cnt);
            if (hist_mass) {
              const uint32_t lo = (uint32_t)run_mass, hi = (uint32_t)(run_mass >> 32);
              const uint32_t old = atomicAdd(&sh.hlo[run_bin], lo);
              const uint32_t carry = (old + lo < old) ? 1u : 0u;
              if (hi + carry) atomicAdd(&sh.hhi[run_bin], hi + carry);
            }
          }
        };
#pragma unroll
        for (int i = 0; i < VE; ++i) {
          if (i >= cnt) break;
          const uint32_t rk = Tr::rkey_of_value(x[i]);
          if (vround || ((rk & hmask) == (prefix & hmask) && rk >= klo && rk <= khi)) {
            const uint32_t bin = vround ? (uint32_t)value_bin(x[i], vb) : ((rk >> shift) & 255u);
            if (!hist_mass) {   // a count-only round: one atomic per element
              atomicAdd(&sh.hcnt[bin], 1u);
              continue;
            }
            if (bin != run_bin) { flush(); run_bin = bin; run_cnt = 0; run_mass = 0; }
            ++run_cnt;
            if (hist_mass) run_mass += mass_fx(ex2_approx((x[i] - M) * c1));
          }
        }
        flush();
        return true;
      });
      ++passes;
      ++rounds;
      __syncthreads();
      if (mass_mode && goal_p >= 0.f && first) {
        unsigned long long tot = 0;
        for (int b = lane; b < 256; b += 32) tot += ((unsigned long long)sh.hhi[b] << 32) + sh.hlo[b];
        tot = warp_sum_u64(tot);
        goal = ceil_mul_frac(goal_p, tot);   // every warp computes the same goal
      }
      if (warp == 0) {
        uint32_t lc = 0;
        unsigned long long lm = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const int b = 255 - 8 * lane - i;
          lc += sh.hcnt[b];
          lm += ((unsigned long long)sh.hhi[b] << 32) + sh.hlo[b];
        }
        uint32_t ic = lc;
        unsigned long long im = lm;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
          const uint32_t yc = __shfl_up_sync(kFullMask, ic, o);
          const unsigned long long ym = __shfl_up_sync(kFullMask, im, o);
          if (lane >= o) { ic += yc; im += ym; }
        }
        const unsigned long long ec = ic - lc, em = im - lm;
        const bool mine_has = mass_mode ? (em < goal && goal <= im) : (ec < goal && goal <= (unsigned long long)ic);
        const uint32_t ballot = __ballot_sync(kFullMask, mine_has);
        if (ballot == 0) {
          if (lane == 0) sh.bsel = 0xFFFFFFFFu;
        } else if (lane == __ffs(ballot) - 1) {
          unsigned long long ac = ec, am = em;
          int sel = -1;
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int b = 255 - 8 * lane - i;
            const unsigned long long cc = sh.hcnt[b], mm = ((unsigned long long)sh.hhi[b] << 32) + sh.hlo[b];
            const bool hit = mass_mode ? (am < goal && goal <= am + mm) : (ac < goal && goal <= ac + cc);
            if (hit && sel < 0) sel = b;
            if (sel < 0) { ac += cc; am += mm; }
          }
          sh.bsel = (uint32_t)sel;
          sh.bq[0] = ac;
          sh.bq[1] = am;
        }
      }
      __syncthreads();
      const uint32_t sel = sh.bsel;
      if (sel > 255u) {
        out.ok = 0;
        return out;
      }
      const unsigned long long ac = sh.bq[0], am = sh.bq[1];
      out.cnt_eq = sh.hcnt[sel];
      out.mass_eq = ((unsigned long long)sh.hhi[sel] << 32) + sh.hlo[sel];
      cnt_above += ac;
      mass_above += am;
      if (mass_mode) goal -= am; else goal -= ac;
      first = false;
      if (vround) {
        // the selected value bin's key range, then key rounds inside it
        const KeyRange kr = key_range_of_bin<Tr>((int)sel, Tr::rkey_of_value(Mmin), Tr::rkey_of_value(M), vb);
        vround = false;
        klo = kr.klo;
        khi = kr.khi;
        prefix = kr.prefix;
        if (kr.shift < 0) break;   // one key: the group
        shift = kr.shift;
        continue;
      }
      prefix |= sel << shift;
      if (shift == 0) break;
      shift -= 8;
    }
    __syncthreads();
    out.rk = prefix;
    out.cnt_above = cnt_above;
    out.mass_above = mass_above;
    out.goal = goal;
    return out;
  }

  // min-p statistics: elements with key >= kmin32 (fp32 key space), their mass, the smallest such key and
  // its count
  __device__ __noinline__ void minp_stats(uint32_t kmin32, uint32_t& cnt_ge, unsigned long long& mass_ge, uint32_t& minkey,
                             uint32_t& cnt_minkey) {
    uint32_t c = 0, mk = 0xFFFFFFFFu, cmk = 0;
    unsigned long long m = 0;
    for_each_tile(0, [&](int64_t, int64_t, const float (&x)[VE], int cnt) {
#pragma unroll
      for (int i = 0; i < VE; ++i) {
        const uint32_t k32 = key_f32_bits(__float_as_uint(x[i]));
        if (i < cnt && k32 >= kmin32) {
          ++c;
          m += mass_fx(ex2_approx((x[i] - M) * c1));
          if (k32 < mk) { mk = k32; cmk = 1; }
          else if (k32 == mk) ++cmk;
        }
      }
      return true;
    });
    ++passes;
    cnt_ge = block_sum_u32(c, sh);
    mass_ge = block_sum_u64(m, sh);
    minkey = block_min_u32(mk, sh);
    cnt_minkey = block_sum_u32(mk == minkey ? cmk : 0u, sh);
  }

  // the index of the need-th element (1-based, index order) equal to xv, visiting vectors from begin_vec;
  // -1 if there are fewer. Tiles of 256 threads x 4 consecutive vectors, one block scan per tile.
  __device__ __noinline__ int32_t nth_equal(float xv, unsigned long long need, int64_t begin_vec) {
    constexpr int PV = 4;
    const unsigned char* xr = p.x + (int64_t)row * p.ld * Tr::ESIZE;
    const int64_t nvec = (n + VE - 1) / VE;
    const int t = threadIdx.x;
    int32_t found = -1;
    unsigned long long before = 0;
    for (int64_t v0 = begin_vec; v0 < nvec; v0 += (int64_t)kSplitThreads * PV) {
      float x[PV][VE];
      int cnt[PV];
      uint32_t c = 0;
#pragma unroll
      for (int q = 0; q < PV; ++q) {
        const int64_t vi = v0 + (int64_t)t * PV + q;
        const int64_t e = vi * VE;
        cnt[q] = vi < nvec ? (n - e >= VE ? VE : (int)(n - e)) : 0;
        if (cnt[q] == VE && p.tma) {
          Tr::values(reinterpret_cast<const uint4*>(xr)[vi], x[q]);
        } else {
#pragma unroll
          for (int i = 0; i < VE; ++i) x[q][i] = i < cnt[q] ? Tr::load_global(xr, e + i) : -INFINITY;
        }
#pragma unroll
        for (int i = 0; i < VE; ++i) c += (i < cnt[q] && x[q][i] == xv) ? 1u : 0u;
      }
      uint32_t tot;
      const uint32_t pre = block_scan_u32(c, tot, sh);
      if (before + pre < need && need <= before + pre + c) {
        unsigned long long seen = before + pre;
#pragma unroll
        for (int q = 0; q < PV; ++q)
#pragma unroll
          for (int i = 0; i < VE; ++i)
            if (i < cnt[q] && x[q][i] == xv && ++seen == need) sh.i[0] = (int32_t)((v0 + (int64_t)t * PV + q) * VE + i);
      }
      const bool done = before + tot >= need;
      before += tot;
      __syncthreads();
      if (done) found = sh.i[0];
      __syncthreads();
      if (done) break;
    }
    ++passes;
    return found;
  }
};

// A piece of a row as one lane sees it: vector u of lane l is vector u * 32 + l of the piece. Aligned rows
// take 16-byte loads; the last, partial vector of a row and unaligned rows are read element by element.
template <typename T>
struct PieceView {
  using Tr = Traits<T>;
  static constexpr int VE = Tr::VE;
  const unsigned char* xr;   // the row
  int64_t V;                 // row length
  int32_t tma;               // the row is 16-byte aligned
  int64_t e_begin;           // first element of the piece
  __device__ __forceinline__ int64_t elem(int u) const {
    return e_begin + (int64_t)(u * 32 + (int)(threadIdx.x & 31)) * VE;
  }
  // the whole piece lies in an aligned row: plain 16-byte loads without bounds
  __device__ __forceinline__ bool full() const { return tma && e_begin + kPieceElems<T> <= V; }
  // start moving the lane's vectors of a full piece towards L1 (the warp's next item, while this one computes)
  __device__ __forceinline__ void prefetch() const {
    if (!full()) return;
    const uint4* b = reinterpret_cast<const uint4*>(xr + e_begin * Tr::ESIZE) + (int)(threadIdx.x & 31);
#pragma unroll
    for (int u = 0; u < kPieceVecs<T>; ++u) asm volatile("prefetch.global.L1 [%0];" ::"l"(b + u * 32));
  }
  __device__ __forceinline__ void get_full(int u, uint4& v) const {
    v = __ldg(reinterpret_cast<const uint4*>(xr + e_begin * Tr::ESIZE) + u * 32 + (int)(threadIdx.x & 31));
  }
  __device__ __forceinline__ int get(int u, uint4& v) const {
    const int64_t e = elem(u);
    const int64_t left = V - e;
    const int cnt = left <= 0 ? 0 : (left >= VE ? VE : (int)left);
    if (cnt == VE && tma) {
      v = __ldg(reinterpret_cast<const uint4*>(xr + e * Tr::ESIZE));
    } else {
      uint32_t w[4] = {0u, 0u, 0u, 0u};
      for (int i = 0; i < cnt; ++i) {
        if (Tr::ESIZE == 4) w[i] = reinterpret_cast<const uint32_t*>(xr)[e + i];
        else w[i >> 1] |= (uint32_t)reinterpret_cast<const uint16_t*>(xr)[e + i] << (16 * (i & 1));
      }
      v = make_uint4(w[0], w[1], w[2], w[3]);
    }
    return cnt;
  }
};

// The index of the need-th element (1-based, index order) equal to xv in a piece; kNoIndex if there are fewer.
// Element order in the piece is (vector u, lane, element i): one warp scan per u. Warp-collective.
template <typename T>
__device__ __noinline__ int32_t piece_nth_equal(const PieceView<T>& pv, float xv, uint32_t need) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  constexpr int U = kPieceVecs<T>;
  const int lane = threadIdx.x & 31;
  uint32_t base = 0;
  int32_t found = kNoIndex;
  for (int u = 0; u < U; ++u) {
    uint4 v;
    const int n = pv.get(u, v);
    float x[VE];
    Tr::values(v, x);
    uint32_t c = 0;
#pragma unroll
    for (int i = 0; i < VE; ++i) c += (i < n && x[i] == xv) ? 1u : 0u;
    uint32_t inc = c;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFullMask, inc, o);
      if (lane >= o) inc += y;
    }
    const uint32_t excl = base + inc - c;
    int32_t idx = kNoIndex;
    if (c && excl < need && need <= excl + c) {
      uint32_t seen = excl;
#pragma unroll
      for (int i = 0; i < VE; ++i)
        if (idx < 0 && i < n && x[i] == xv && ++seen == need) idx = (int32_t)(pv.elem(u) + i);
    }
    const uint32_t hit = __ballot_sync(kFullMask, idx >= 0);
    if (hit) {
      found = __shfl_sync(kFullMask, idx, __ffs(hit) - 1);
      break;
    }
    base += __shfl_sync(kFullMask, inc, 31);
  }
  return found;
}

// ------------------------------------------------------------------------------------------------
// The streaming sampler (vsamp_sample_ws, vsamp_sample_static): two launches, no waiting inside either.
//   piece_kernel   every warp takes 4 KB pieces of the batch, grid-stride, each arriving in shared memory by a
//                  bulk copy issued one piece ahead (plain loads for a partial piece or an unaligned row). It
//                  writes the piece's record: maximum, minimum, count of maxima and mass relative to its maximum
//                  (2^-40 fixed point per 16-byte vector). For a row that draws over a possibly large kept set
//                  (no top-k, T > 0) it also forms every token's Philox word (the words depend only on (seed,
//                  row_id, step), not on the logits) and writes a 4-bit draw code per vector.
//   row_kernel     one CTA per row combines the row's piece records in a fixed order, plans the cut (radix rounds
//                  re-read the row from L2 only when the cut leaves the maximum's tie group), and draws: in every
//                  piece that holds a kept token, the vectors whose code passes the row's prune bound are read
//                  again and scored exactly; rows without codes scan their kept tokens. It writes the outputs.
// Per row the result is a function of the row alone (pieces are fixed by V, combined in a fixed order). Every
// call writes the workspace before reading it, so the workspace needs no initialisation.
// ------------------------------------------------------------------------------------------------
struct StreamHeader {                // the first 256 bytes of the workspace (reserved)
  uint32_t reserved[64];
};
static_assert(sizeof(StreamHeader) == 256, "StreamHeader layout");

struct PieceRec {                    // 32 bytes per (row, piece)
  float m;                           // piece maximum (NaN: a non-finite value, or the load timed out)
  uint32_t cnt;                      // elements equal to m (kTimeoutCnt when the load timed out)
  unsigned long long s;              // sum of 2^((x - m) * c1), 2^-40 fixed point
  float mn;                          // piece minimum
  uint32_t reserved[3];
};
static_assert(sizeof(PieceRec) == 32, "PieceRec layout");

constexpr int kItemPieces = kStreamThreads / 32;   // warps per CTA
constexpr uint32_t kTimeoutCnt = 0xFFFFFFFFu;
constexpr int kFlagMax = 1024;                     // flagged vectors a row finish collects before it scans instead

struct StreamWs {
  PieceRec* recs;                    // [B, rec_ld]: the first np records of each row
  int64_t rec_ld;                    // records per row in `recs` (np, or more for a shard's record slots)
  uint32_t* codes;                   // [B, np, 32]: lane l's word holds the codes of vectors u * 32 + l
};

// Workspace bytes: header | PieceRec[B, np] | codes[B, np, 32].
inline size_t split_workspace_bytes(int64_t B, int64_t V, int esize) {
  const size_t np = (size_t)split_nchunks(V, esize);
  return sizeof(StreamHeader) + (size_t)B * np * sizeof(PieceRec) + (size_t)B * np * 32u * sizeof(uint32_t);
}

// A piece record written by the other launch: read through L2 (kLocal: a record in this CTA's shared memory).
template <bool kLocal = false>
__device__ __forceinline__ PieceRec load_rec(const PieceRec* a) {
  const uint4 v0 = kLocal ? reinterpret_cast<const uint4*>(a)[0] : __ldcg(reinterpret_cast<const uint4*>(a));
  const uint4 v1 = kLocal ? reinterpret_cast<const uint4*>(a)[1] : __ldcg(reinterpret_cast<const uint4*>(a) + 1);
  PieceRec r;
  r.m = __uint_as_float(v0.x);
  r.cnt = v0.y;
  r.s = ((unsigned long long)v0.w << 32) | v0.z;
  r.mn = __uint_as_float(v1.x);
  return r;
}

// Shared memory of a piece_kernel CTA: per warp, two 4 KB piece buffers and their mbarriers.
struct PieceSmem {
  unsigned long long bar[kItemPieces][2];
  __align__(128) uint4 buf[kItemPieces][2][kPieceBytes / 16];
};

constexpr int kCodeSmem = 4800;   // code words a row finish stages in shared memory: rows of up to 150 pieces

// Shared memory of a row_kernel CTA.
struct FinishSmem {
  SplitShared sh;
  int32_t it;                                          // the cut's last kept index
  uint32_t nflag;                                      // flagged vectors
  float bs[kItemPieces], bsv[kItemPieces];             // per-warp best score, its scaled logit
  int32_t bi[kItemPieces];                             //   and index
  uint32_t flist[kFlagMax];                            // flagged vector indices
  uint32_t codes[kCodeSmem];                           // the row's draw codes
  __align__(16) uint4 piece[kPieceBytes / 16];         // the boundary piece
};

// The parameters of one row's draw.
struct DrawRow {
  float M, invT, c1, xP, kappa;
  int32_t It;
  uint32_t bk, rid, st_lo, st_hi;
  PhiloxKey key;
  bool all_cand;
};

// Exact perturbed scores of one vector's kept tokens that pass the prune bound (every kept token when all
// kept tokens are candidates); the running arg-max (score, index, scaled logit) is updated in place.
template <typename T>
__device__ __noinline__ void score_vector(uint4 v, int cnt, int64_t e0, const DrawRow& d, float& bscore, int32_t& bidx,
                                          float& bs) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  float x[VE];
  Tr::values(v, x);
  uint32_t kmask = 0u;
#pragma unroll
  for (int i = 0; i < VE; ++i)
    if (i < cnt && (x[i] > d.xP || (x[i] == d.xP && e0 + i <= (int64_t)d.It))) kmask |= 1u << i;
  if (!kmask) return;
  uint32_t b[VE];
#pragma unroll
  for (int g = 0; g < VE / 4; ++g) {
    const uint4 w4 = philox4x32_10(make_uint4((uint32_t)(e0 >> 2) + (uint32_t)g, d.rid, d.st_lo, d.st_hi), d.key);
    b[4 * g + 0] = w4.x; b[4 * g + 1] = w4.y; b[4 * g + 2] = w4.z; b[4 * g + 3] = w4.w;
  }
#pragma unroll
  for (int i = 0; i < VE; ++i) {
    if (!((kmask >> i) & 1u)) continue;
    if (!d.all_cand && b[i] >= d.bk) continue;
    const float dx = x[i] - d.M;
    const float sv = dx * d.invT;
    if (!d.all_cand) {
      const float w = ex2_approx(dx * d.c1);
      const float u = fmaf((float)b[i], kTwoM32, kTwoM33);
      if (!(u < w * d.kappa * 1.00001f)) continue;
    }
    const float score = gumbel_score(sv, b[i]);
    const int32_t idx = (int32_t)(e0 + i);
    if (argmax_better(score, idx, bscore, bidx)) { bscore = score; bidx = idx; bs = sv; }
  }
}

// Every kept token of a row scored (pruned unless all are candidates), the row read from L2: each thread takes
// vectors t, t + 256, ... (rows drawn without codes, and the certification fallback).
template <typename T>
__device__ __noinline__ void score_row(const Params& p, int64_t row, const DrawRow& d, float& bscore, int32_t& bidx,
                                       float& bs) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  const unsigned char* xr = p.x + row * p.ld * Tr::ESIZE;
  const int64_t nvec = (p.V + VE - 1) / VE;
  for (int64_t vi = threadIdx.x; vi < nvec; vi += kStreamThreads) {
    uint4 v;
    const int cnt = load_vec<T, false>(p, xr, vi * VE, v);
    score_vector<T>(v, cnt, p.v0 + vi * VE, d, bscore, bidx, bs);   // global index: counters and the result
  }
}

// The CTA's arg-max of (score, index), ties to the lower index; every thread gets it.
__device__ __forceinline__ ArgMax block_argmax(ArgMax a, FinishSmem& S) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  a = warp_argmax(a);
  __syncthreads();
  if (lane == 0) { S.bs[warp] = a.score; S.bi[warp] = a.idx; S.bsv[warp] = a.s; }
  __syncthreads();
  ArgMax b{S.bs[0], S.bi[0], S.bsv[0]};
#pragma unroll
  for (int w = 1; w < kItemPieces; ++w)
    if (argmax_better(S.bs[w], S.bi[w], b.score, b.idx)) b = ArgMax{S.bs[w], S.bi[w], S.bsv[w]};
  return b;
}

// A row draws with codes when its parameters allow a large kept set: sampled (T > 0) and no top-k.
__device__ __forceinline__ bool row_coded(const Params& p, int64_t row) {
  const float temp0 = p.temperature ? p.temperature[row] : 1.f;
  const int32_t topk = p.top_k ? p.top_k[row] : 0;
  return temp0 > 0.f && !(topk > 0 && (int64_t)topk < p.V);
}

// The index of the need-th element (1-based, index order) equal to xv in a piece, kNoIndex if there are fewer.
// One warp: the piece is staged in shared memory (all of the lane's loads issued at once), then scanned in the
// piece's order (vector u, lane, element) with compact loops.
template <typename T>
__device__ __noinline__ int32_t piece_nth_equal_staged(const PieceView<T>& pv, float xv, uint32_t need, uint4* stage) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  constexpr int U = kPieceVecs<T>;
  const int lane = threadIdx.x & 31;
  int n[U];
  {
    uint4 v[U];
#pragma unroll
    for (int u = 0; u < U; ++u) n[u] = pv.get(u, v[u]);
#pragma unroll
    for (int u = 0; u < U; ++u) stage[u * 32 + lane] = v[u];
  }
  const int64_t left = pv.V - pv.e_begin;   // valid elements of the piece (its vectors past them count nothing)
  __syncwarp();
  uint32_t base = 0;
#pragma unroll 1
  for (int u = 0; u < U; ++u) {
    float x[VE];
    Tr::values(stage[u * 32 + lane], x);
    const int64_t e_in = (int64_t)(u * 32 + lane) * VE;
    const int cnt = left - e_in >= VE ? VE : (left - e_in > 0 ? (int)(left - e_in) : 0);
    uint32_t c = 0;
#pragma unroll 1
    for (int i = 0; i < cnt; ++i) c += x[i] == xv ? 1u : 0u;
    uint32_t inc = c;
#pragma unroll 1
    for (int o = 1; o < 32; o <<= 1) {
      const uint32_t y = __shfl_up_sync(kFullMask, inc, o);
      if (lane >= o) inc += y;
    }
    const uint32_t excl = base + inc - c;
    int32_t idx = kNoIndex;
    if (c && excl < need && need <= excl + c) {
      uint32_t seen = excl;
#pragma unroll 1
      for (int i = 0; i < cnt; ++i)
        if (x[i] == xv && ++seen == need) { idx = (int32_t)(pv.e_begin + e_in + i); break; }
    }
    const uint32_t hit = __ballot_sync(kFullMask, idx >= 0);
    if (hit) return __shfl_sync(kFullMask, idx, __ffs(hit) - 1);
    base += __shfl_sync(kFullMask, inc, 31);
  }
  (void)n;
  return kNoIndex;
}

// ------------------------------------------------------------------------------------------------
// The cut of one row (a CTA): the shortest prefix of the order (value desc, index asc) over top-k, top-p (on
// the top-k mass) and min-p, at least one token. From the row statistics (maximum P.M, fixed-point mass Sfx,
// count of maxima cM); radix rounds and the min-p pass re-read the row through the planner only when the cut
// leaves the maximum's tie group. Sets PATH_* flags in `path` and a row error in `plan_status`.
// ------------------------------------------------------------------------------------------------
template <typename T>
static __device__ __noinline__ Cut plan_cut(RowPlanner<T>& P, bool greedy, float Teff, int32_t topk, float topp,
                                            float minp, unsigned long long Sfx, uint32_t cM, int& path,
                                            int& plan_status) {
  using Tr = Traits<T>;
  const int64_t n = P.n;
  const float M = P.M, c1 = P.c1;
  const unsigned long long one = 1ull << kMassShift;
  const uint32_t rkM = Tr::rkey_of_value(M);
  Cut fin{};
  bool minp_on = !greedy && minp > 0.f;
  if (greedy) {
    fin = Cut{rkM, 0, 1, cM, one, 0};
    path |= PATH_MAXGROUP;
  } else {
    int ck_mode = 0, cp_mode = 0;
    float goal_p = -1.f;
    unsigned long long cp_goal = 0ull;
    Cut ck{}, cp{};
    const bool topk_on = topk > 0 && (int64_t)topk < n;
    const bool topp_on = topp < 1.f;
    const unsigned long long keff = topk_on ? (unsigned long long)topk : (unsigned long long)n;
    if (topk_on) {
      if (keff <= cM) { ck = Cut{rkM, 0, keff, cM, keff * one, 0}; ck_mode = 1; }
      else { ck = Cut{0, 0, keff, 0, 0, 0}; ck_mode = 2; }
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
    // top-p keeping the first maximum alone is the shortest cut: no radix search for top-k, no min-p pass
    const bool cp_one = cp_mode == 1 && cp.kept() == 1;
    if (cp_one && ck_mode == 2) ck_mode = 0;
    if (ck_mode == 1 || cp_mode == 1) path |= PATH_MAXGROUP;
    if (minp_on && !cp_one) {
      // min-p keeps w >= minp <=> x >= x* = M + T ln(minp) (an unevaluated sum; the threshold is the
      // smallest fp32 value >= x*): the kept group ends with the smallest key at or above it
      const float L = logf(minp);
      const float ph = Teff * L, pl_ = fmaf(Teff, L, -ph);
      const float sh_ = M + ph;
      const float bb = sh_ - M;
      const float sl = (M - (sh_ - bb)) + (ph - bb);
      const float lo = sl + pl_;
      const float xf = lo > 0.f ? nextafterf(sh_, INFINITY) : sh_;
      const uint32_t kmin32 = key_f32_bits(__float_as_uint(xf));
      // a threshold at or below the row's minimum keeps every token: the filter is off (no pass)
      if (kmin32 <= key_f32_bits(__float_as_uint(P.Mmin))) minp_on = false;
      if (minp_on) {
        uint32_t cnt_ge, minkey, cnt_minkey;
        unsigned long long mass_ge;
        P.minp_stats(kmin32, cnt_ge, mass_ge, minkey, cnt_minkey);
        const uint32_t rkm = (Tr::KB == 32) ? minkey : (minkey >> 16);
        fin = Cut{rkm, (unsigned long long)(cnt_ge - cnt_minkey), cnt_minkey, cnt_minkey, mass_ge, 1};
      }
    }
    if (!(minp_on && !cp_one)) {
      fin = Cut{rkM, 0, (unsigned long long)n, 0, Sfx, 1};
    }
    if (ck_mode == 2) {
      const RadixOut r = P.radix(false, ck.need, -1.f, cp_mode == 2);
      if (!r.ok) plan_status = VSAMP_ERR_INVALID_ARG;
      const unsigned long long need = ck.need - r.cnt_above;
      const unsigned long long wP = mass_fx(ex2_approx((Tr::value_of_rkey(r.rk) - M) * c1));
      ck = Cut{r.rk, r.cnt_above, need, r.cnt_eq, r.mass_above + need * wP, 0};
      path |= PATH_RADIX_K;
      if (cp_mode == 2) cp_goal = ceil_mul_frac(topp, ck.mass);
    }
    if (cp_mode == 2 && plan_status == VSAMP_OK) {
      const RadixOut r = P.radix(true, cp_goal, goal_p, true);
      if (!r.ok) plan_status = VSAMP_ERR_INVALID_ARG;
      const unsigned long long wP = mass_fx(ex2_approx((Tr::value_of_rkey(r.rk) - M) * c1));
      unsigned long long need = wP ? (r.goal + wP - 1) / wP : 1;
      need = need < 1 ? 1 : (need > r.cnt_eq ? r.cnt_eq : need);
      cp = Cut{r.rk, r.cnt_above, need, r.cnt_eq, r.mass_above + need * wP, 0};
      path |= PATH_RADIX_P;
    }
    Cut best = fin;
    if (ck_mode && ck.kept() < best.kept()) best = ck;
    if (cp_mode && cp.kept() < best.kept()) best = cp;
    if (minp_on && best.whole) path |= PATH_MINP;
    fin = best;
  }
  return fin;
}

// ------------------------------------------------------------------------------------------------
// Row finish: one CTA (all 256 threads) per row. The row's dependent memory accesses are batched: the piece
// records and the draw codes come in one round of loads, and after the plan the boundary piece and the flagged
// vectors in another. kLocal: the records (ws.recs, rec_ld 0) and the codes (S.codes) are already in this
// CTA's shared memory.
// ------------------------------------------------------------------------------------------------
template <typename T, bool kLocal = false>
static __device__ __forceinline__ void finish_row(const Params& p, const StreamWs& ws, int64_t row, int nchunks,
                                                  FinishSmem& S) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  SplitShared& sh = S.sh;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t n = p.V;
  const PieceRec* recs = ws.recs + row * ws.rec_ld;
  const float temp0 = p.temperature ? p.temperature[row] : 1.f;
  const float Teff = temp0 > 0.f ? temp0 : 1.f;   // greedy rows use T = 1 for their statistics
  const float invT = 1.f / Teff;
  const float c1 = kLog2e * invT;
  const bool coded = row_coded(p, row);
  const int64_t nwords = (int64_t)nchunks * 32;
  const bool codes_staged = coded && nwords <= (int64_t)kCodeSmem;
  // ---- one round of loads: the thread's first two piece records and the row's codes into shared memory ----
  PieceRec r0{}, r1{};
  if (t < nchunks) r0 = load_rec<kLocal>(recs + t);
  if (t + kStreamThreads < nchunks) r1 = load_rec<kLocal>(recs + t + kStreamThreads);
  if (codes_staged && !kLocal) {
    const uint32_t* src = ws.codes + row * nwords;
#pragma unroll 4
    for (int w = t; w < (int)nwords; w += kStreamThreads) S.codes[w] = __ldcg(src + w);
  }
  auto rec_at = [&](int k) -> PieceRec {
    return k == t ? r0 : (k == t + kStreamThreads ? r1 : load_rec<kLocal>(recs + k));
  };
  // ---- combine the pieces: M and the flags, then S rescaled to M and the count of maxima ----
  float m = -INFINITY, mn = INFINITY;
  uint32_t flags = 0;   // 1: a non-finite value, 2: a load timed out
  for (int k = t; k < nchunks; k += kStreamThreads) {
    const PieceRec r = rec_at(k);
    if (r.m != r.m) flags |= r.cnt == kTimeoutCnt ? 3u : 1u;
    else { m = fmaxf(m, r.m); mn = fminf(mn, r.mn); }
  }
  m = warp_max_f(m);
  mn = -warp_max_f(-mn);
  flags = __reduce_or_sync(kFullMask, flags);
  if (lane == 0) { sh.f[warp] = m; sh.u[warp][0] = flags; sh.u[warp][2] = __float_as_uint(mn); }
  __syncthreads();
  float M = sh.f[0], Mmin = __uint_as_float(sh.u[0][2]);
  flags = sh.u[0][0];
#pragma unroll
  for (int w = 1; w < kItemPieces; ++w) {
    M = fmaxf(M, sh.f[w]);
    Mmin = fminf(Mmin, __uint_as_float(sh.u[w][2]));
    flags |= sh.u[w][0];
  }
  const bool nonfin = flags != 0u;
  unsigned long long Sp = 0;
  uint32_t cMp = 0;
  for (int k = t; k < nchunks; k += kStreamThreads) {
    const PieceRec r = rec_at(k);
    if (r.m == M) {
      Sp += r.s;
      cMp += r.cnt;
    } else if (!nonfin) {
      // 2^((m_p - M) * c1) is below 1: the piece's fixed-point mass rescaled in binary64
      const double f = exp2((double)((r.m - M) * c1));
      Sp += (unsigned long long)__double2ull_rn((double)r.s * f);
    }
  }
  Sp = warp_sum_u64(Sp);
  cMp = warp_sum_u32(cMp);
  if (lane == 0) { sh.q[warp][0] = Sp; sh.u[warp][1] = cMp; }
  __syncthreads();
  unsigned long long Sfx = 0;
  uint32_t cM = 0;
#pragma unroll
  for (int w = 0; w < kItemPieces; ++w) { Sfx += sh.q[w][0]; cM += sh.u[w][1]; }

  // ---- status ----
  const float topp = p.top_p ? p.top_p[row] : 1.f;
  const float minp = p.min_p ? p.min_p[row] : 0.f;
  const int32_t topk = p.top_k ? p.top_k[row] : 0;
  int status = VSAMP_OK;
  if (flags & 2u) status = VSAMP_ERR_TIMEOUT;
  else if (flags) status = VSAMP_ERR_NONFINITE;
  else if (isnan(temp0) || isinf(temp0) || isnan(topp) || !(topp > 0.f) || isnan(minp) || minp > 1.f)
    status = VSAMP_ERR_INVALID_ARG;
  const bool greedy = !(temp0 > 0.f);
  int path = p.tma ? 0 : PATH_NOTMA;
  RowPlanner<T> P{p, sh, row, n, M, c1};
  P.Mmin = Mmin;
  P.passes = 1;
  auto write_outputs = [&](int32_t tok, float lp, int st, uint32_t kept) {
    if (t == 0) {
      p.token[row] = tok;
      if (p.logprob) p.logprob[row] = lp;
      if (p.row_status) p.row_status[row] = st;
      if (p.stats) {
        p.stats[row * 4 + 0] = P.passes;
        p.stats[row * 4 + 1] = P.rounds;
        p.stats[row * 4 + 2] = (int32_t)kept;
        p.stats[row * 4 + 3] = path;
      }
    }
  };
  if (status != VSAMP_OK) {
    write_outputs(-1, __int_as_float(0x7FC00000), status, 0u);
    return;
  }
  const float logS = logf(u64_to_float(Sfx) * 9.094947017729282379e-13f);   // 2^-40
  const unsigned long long one = 1ull << kMassShift;
  const uint32_t rkM = Tr::rkey_of_value(M);

  // ---- plan: the shortest prefix over top-k, top-p and min-p ----
  int plan_status = VSAMP_OK;
  const Cut fin = plan_cut<T>(P, greedy, Teff, topk, topp, minp, Sfx, cM, path, plan_status);
  if (plan_status != VSAMP_OK) {
    write_outputs(-1, __int_as_float(0x7FC00000), plan_status, 0u);
    return;
  }

  // ---- the cut, the prune bound, and the flagged vectors ----
  const unsigned long long kept = fin.kept();
  const bool one_token = greedy || kept == 1;
  float xP = Tr::value_of_rkey(fin.rk);
  const float skept = fmaxf(u64_to_float(fin.mass) * 9.094947017729282379e-13f, 1.f);
  DrawRow d;
  d.M = M;
  d.invT = invT;
  d.c1 = c1;
  d.kappa = 20.085536923187668f / skept;
  d.all_cand = d.kappa >= 0.99f;
  d.bk = d.all_cand ? 0xFFFFFFFFu : __float2uint_ru(d.kappa * 1.00001f * 4294967296.0f);
  // the flagged vectors of a coded row, from the staged codes (their loads do not need the cut's index)
  const bool from_codes = !one_token && codes_staged && !d.all_cand;
  uint32_t nflag = 0;
  if (from_codes) {
    if (t == 0) S.nflag = 0u;
    __syncthreads();   // also: the staged codes are visible
    const uint32_t cbk = draw_code(d.bk);
    const int64_t nvec = (n + VE - 1) / VE;
    // nibbles >= cbk, eight at a time: even and odd nibbles in separate bytes, so adding 16 - cbk carries into
    // bit 4 of a byte exactly when its nibble is >= cbk
    const uint32_t addk = (16u - cbk) * 0x01010101u;
#pragma unroll 1
    for (int w = t; w < (int)nwords; w += kStreamThreads) {
      const uint32_t word = S.codes[w];
      const uint32_t ge = (((word & 0x0F0F0F0Fu) + addk) & 0x10101010u) | ((((word >> 4) & 0x0F0F0F0Fu) + addk) & 0x10101010u);
      if (!ge && cbk) continue;
#pragma unroll 1
      for (int u = 0; u < kPieceVecs<T>; ++u) {
        if (((word >> (4 * u)) & 15u) < cbk) continue;
        const int64_t vi = (int64_t)(w >> 5) * (kPieceElems<T> / VE) + u * 32 + (w & 31);
        if (vi >= nvec) continue;
        const uint32_t slot = atomicAdd(&S.nflag, 1u);
        if (slot < (uint32_t)kFlagMax) S.flist[slot] = (uint32_t)vi;
      }
    }
    __syncthreads();
    nflag = S.nflag;
  }
  // this thread's first flagged vector, loaded now (the boundary search below runs meanwhile)
  const unsigned char* xr = p.x + row * p.ld * Tr::ESIZE;
  uint4 fv = make_uint4(0u, 0u, 0u, 0u);
  int fcnt = 0;
  int64_t fe0 = 0;
  const bool have_f = from_codes && nflag <= (uint32_t)kFlagMax && (uint32_t)t < nflag;
  if (have_f) {
    fe0 = (int64_t)S.flist[t] * VE;
    fcnt = load_vec<T, false>(p, xr, fe0, fv);
  }
  int32_t It = kAllIndex;
  if (fin.whole && !one_token) {
    if (fin.above == 0 && fin.cnt_eq == 0) xP = -INFINITY;   // every element
  } else if (fin.rk == rkM) {
    // the need-th maximum: its piece from the piece counts, then one warp scans that piece
    const unsigned long long need = fin.whole ? cM : fin.need;
    unsigned long long before = 0;
    int64_t cb = -1;
    for (int64_t k0 = 0; k0 < nchunks && cb < 0; k0 += kStreamThreads) {
      const int64_t k = k0 + t;
      uint32_t ck = 0;
      if (k < nchunks) {
        const PieceRec r = rec_at((int)k);
        ck = r.m == M ? r.cnt : 0u;
      }
      uint32_t tot;
      const uint32_t pre = block_scan_u32(ck, tot, sh);
      if (before + pre < need && need <= before + pre + ck) {
        sh.bq[2] = (unsigned long long)k;
        sh.bq[3] = before + pre;
      }
      const bool done = before + tot >= need;
      before += tot;
      __syncthreads();
      if (done) cb = (int64_t)sh.bq[2];
      __syncthreads();
    }
    if (warp == 0) {
      int32_t found = kNoIndex;
      if (cb >= 0) {
        const PieceView<T> pv{xr, n, p.tma, cb * kPieceElems<T>};
        found = piece_nth_equal_staged<T>(pv, M, (uint32_t)(need - sh.bq[3]), S.piece);
      }
      if (lane == 0) S.it = found;
    }
    __syncthreads();
    It = S.it;
    ++P.passes;
  } else {
    const unsigned long long need = fin.whole ? fin.cnt_eq : fin.need;
    It = P.nth_equal(xP, need, 0);
  }
  if (It < 0) {   // cannot happen with consistent counts; reported as an error
    write_outputs(-1, __int_as_float(0x7FC00000), VSAMP_ERR_INVALID_ARG, 0u);
    return;
  }
  if (one_token) {
    // the first maximum; (x - M) / T = 0
    write_outputs(It, fminf(-logS, 0.f), VSAMP_OK, (uint32_t)kept);
    return;
  }

  // ---- the draw: a token can beat B0 = ln(S_kept) - 3 only if u < w * kappa ----
  d.xP = xP;
  d.It = It;
  const uint64_t sd = p.seed ? p.seed[row] : 0ull;
  const uint64_t stp = p.step ? p.step[row] : 0ull;
  d.rid = p.row_id ? p.row_id[row] : (uint32_t)row;
  d.st_lo = (uint32_t)stp;
  d.st_hi = (uint32_t)(stp >> 32);
  d.key = PhiloxKey{(uint32_t)sd, (uint32_t)(sd >> 32)};
  const float B0 = -logf(d.kappa);
  float bscore = -INFINITY, bs = 0.f;
  int32_t bidx = 0x7FFFFFFF;
  if (from_codes && nflag <= (uint32_t)kFlagMax) {
    if (have_f) score_vector<T>(fv, fcnt, fe0, d, bscore, bidx, bs);
    for (uint32_t i = t + kStreamThreads; i < nflag; i += kStreamThreads) {
      const int64_t e0 = (int64_t)S.flist[i] * VE;
      uint4 v;
      const int cnt = load_vec<T, false>(p, xr, e0, v);
      score_vector<T>(v, cnt, e0, d, bscore, bidx, bs);
    }
  } else {
    score_row<T>(p, row, d, bscore, bidx, bs);
  }
  ++P.passes;
  ArgMax g = block_argmax(ArgMax{bscore, bidx, bs}, S);
  if (!(d.all_cand || (g.idx != 0x7FFFFFFF && g.score > B0 + 1e-4f * fmaxf(1.f, fabsf(B0))))) {
    // the prune bound did not certify the draw (probability ~1e-9): every kept token of the row, exactly
    path |= PATH_FALLBACK;
    DrawRow all = d;
    all.all_cand = true;
    bscore = -INFINITY;
    bs = 0.f;
    bidx = 0x7FFFFFFF;
    score_row<T>(p, row, all, bscore, bidx, bs);
    g = block_argmax(ArgMax{bscore, bidx, bs}, S);
  }
  if (g.idx >= 0 && (int64_t)g.idx < n) write_outputs(g.idx, fminf(g.s - logS, 0.f), VSAMP_OK, (uint32_t)kept);
  else write_outputs(-1, __int_as_float(0x7FC00000), VSAMP_ERR_INVALID_ARG, 0u);
}

// ------------------------------------------------------------------------------------------------
// Draw codes of one piece: the smallest Philox word of each of the lane's vectors, four counters at a time. The
// words do not depend on the logits; vectors past the row's end get codes too (their tokens are never kept).
// ------------------------------------------------------------------------------------------------
template <typename T>
static __device__ __forceinline__ void piece_codes(int64_t e_begin, uint32_t k0, uint32_t k1, uint32_t rid,
                                                   uint32_t st_lo, uint32_t st_hi, uint32_t* code_out) {
  constexpr int VE = Traits<T>::VE;
  constexpr int U = kPieceVecs<T>;
  constexpr int G = VE / 4;            // Philox counters per vector
  const int lane = threadIdx.x & 31;
  const PhiloxRowMin ph(PhiloxKey{k0, k1}, rid, st_lo, st_hi);
  // counter of group g of vector u: (first element of the piece) / 4 + (u * 32 + lane) * G + g
  const uint32_t cb0 = (uint32_t)(e_begin >> 2) + (uint32_t)(lane * G);
  uint32_t word = 0u;
#pragma unroll 1
  for (int u0 = 0; u0 < U; u0 += 4 / G) {
    uint32_t c[4], mw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) c[i] = cb0 + (uint32_t)((u0 + i / G) * 32 * G + i % G);
    ph.min_words<4>(c, mw);
#pragma unroll
    for (int q = 0; q < 4 / G; ++q) {
      uint32_t mu = mw[q * G];
#pragma unroll
      for (int g = 1; g < G; ++g) mu = min(mu, mw[q * G + g]);
      word |= draw_code(mu) << (4 * (u0 + q));
    }
  }
  code_out[lane] = word;
}

// ------------------------------------------------------------------------------------------------
// Statistics of a partial piece, or of a piece of an unaligned row: the lanes' vectors from global memory, with
// element counts per vector (out of line: the full-piece path keeps its registers). No winner, no codes.
// kHeadOnly: only the record's first 16 bytes {m, cnt, s} are written (the piece minimum is left out).
// ------------------------------------------------------------------------------------------------
template <typename T, bool kHeadOnly = false>
static __device__ __noinline__ void piece_stats_partial(const unsigned char* xr, int64_t V, int32_t tma,
                                                        int64_t e_begin, float c1, bool timeout, PieceRec* rec_out) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  constexpr int U = kPieceVecs<T>;
  const int lane = threadIdx.x & 31;
  uint4 v[U];
  int cnt[U];
  const PieceView<T> pv{xr, V, tma, e_begin};
#pragma unroll
  for (int u = 0; u < U; ++u) cnt[u] = pv.get(u, v[u]);
  float mt = -INFINITY, mn = INFINITY, nf = 0.f;
#pragma unroll
  for (int u = 0; u < U; ++u) {
    float x[VE];
    Tr::values(v[u], x);
#pragma unroll
    for (int i = 0; i < VE; ++i)
      if (i < cnt[u]) { mt = fmaxf(mt, x[i]); mn = fminf(mn, x[i]); nf = fmaf(x[i], 0.f, nf); }
  }
  const float mc = warp_max_f(mt);
  mn = -warp_max_f(-mn);
  const bool bad = timeout || __any_sync(kFullMask, nf != 0.f);
  unsigned long long s = 0ull;
  uint32_t cm = 0u;
  if (!bad) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (cnt[u] <= 0) continue;
      float x[VE], w[VE];
      Tr::values(v[u], x);
      if (cnt[u] == VE) {
        // the same order of additions as a full vector
        const float2 mM = make_float2(-mc, -mc), cc = make_float2(c1, c1);
        float2 w2[VE / 2];
#pragma unroll
        for (int h = 0; h < VE / 2; ++h) {
          const float2 e = __fmul2_rn(__fadd2_rn(make_float2(x[2 * h], x[2 * h + 1]), mM), cc);
          w2[h] = make_float2(ex2_approx(e.x), ex2_approx(e.y));
        }
        float2 a;
        if constexpr (VE == 8) a = __fadd2_rn(__fadd2_rn(w2[0], w2[2]), __fadd2_rn(w2[1], w2[3]));
        else a = __fadd2_rn(w2[0], w2[1]);
        s += mass_fx(a.x + a.y);
#pragma unroll
        for (int i = 0; i < VE; ++i) cm += x[i] == mc ? 1u : 0u;
      } else {
#pragma unroll
        for (int i = 0; i < VE; ++i) {
          const bool ok = i < cnt[u];
          const float d = x[i] - mc;
          w[i] = ok ? ex2_approx(d * c1) : 0.f;
          cm += (ok && d == 0.f) ? 1u : 0u;
        }
#pragma unroll
        for (int h = VE / 2; h >= 1; h >>= 1)
#pragma unroll
          for (int i = 0; i < h; ++i) w[i] += w[i + h];
        s += mass_fx(w[0]);
      }
    }
  }
  s = warp_sum_u64(s);
  cm = warp_sum_u32(cm);
  if (lane == 0) {
    uint4* o = reinterpret_cast<uint4*>(rec_out);
    o[0] = make_uint4(bad ? 0x7FC00000u : __float_as_uint(mc), timeout ? kTimeoutCnt : cm, (uint32_t)s, (uint32_t)(s >> 32));
    if (!kHeadOnly) o[1] = make_uint4(__float_as_uint(mn), 0u, 0u, 0u);
  }
}

// ------------------------------------------------------------------------------------------------
// Piece pass of one warp over a full piece in shared memory: the record, and for a coded row the draw codes
// (e_begin: the global index of the piece's first element, for the Philox counters). kHeadOnly: only the
// record's head {m, 0, s}, without the piece minimum and the count of maxima (the row statistics alone).
// ------------------------------------------------------------------------------------------------
template <typename T, bool kHeadOnly = false>
static __device__ __forceinline__ void piece_pass_full(const uint4* sbuf, int64_t e_begin, float c1,
                                                       bool timeout, bool coded, uint32_t k0, uint32_t k1,
                                                       uint32_t rid, uint32_t st_lo, uint32_t st_hi,
                                                       PieceRec* rec_out, uint32_t* code_out) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  constexpr int U = kPieceVecs<T>;     // vectors per lane and piece: 8
  constexpr int G = VE / 4;            // Philox counters per vector
  const int lane = threadIdx.x & 31;
  // ---- maximum, minimum, non-finite check ----
  float mt, mn, nf;
  if constexpr (VE == 8) {
    const __nv_bfloat162 zero2 = __float2bfloat162_rn(0.f);
    __nv_bfloat162 mx2 = __float2bfloat162_rn(-INFINITY), mn2 = __float2bfloat162_rn(INFINITY), nf2 = zero2;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint4 v = sbuf[u * 32 + lane];
      const __nv_bfloat162 a = Tr::pair(v.x), b = Tr::pair(v.y), c = Tr::pair(v.z), d = Tr::pair(v.w);
      mx2 = __hmax2(mx2, __hmax2(__hmax2(a, b), __hmax2(c, d)));
      if (!kHeadOnly) mn2 = __hmin2(mn2, __hmin2(__hmin2(a, b), __hmin2(c, d)));
      nf2 = __hfma2(a, zero2, __hfma2(b, zero2, __hfma2(c, zero2, __hfma2(d, zero2, nf2))));
    }
    mt = fmaxf(__low2float(mx2), __high2float(mx2));
    mn = fminf(__low2float(mn2), __high2float(mn2));
    nf = (__low2float(nf2) != 0.f || __high2float(nf2) != 0.f) ? 1.f : 0.f;
  } else {
    mt = -INFINITY;
    mn = INFINITY;
    nf = 0.f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float x[VE];
      Tr::values(sbuf[u * 32 + lane], x);
      mt = fmaxf(mt, fmaxf(fmaxf(x[0], x[1]), fmaxf(x[2], x[3])));
      if (!kHeadOnly) mn = fminf(mn, fminf(fminf(x[0], x[1]), fminf(x[2], x[3])));
      nf = fmaf(x[0], 0.f, fmaf(x[1], 0.f, fmaf(x[2], 0.f, fmaf(x[3], 0.f, nf))));
    }
  }
  const float mc = warp_max_f(mt);
  if (!kHeadOnly) mn = -warp_max_f(-mn);
  const bool bad = timeout || __any_sync(kFullMask, nf != 0.f);
  // ---- mass relative to the piece maximum (2^-40 fixed point per vector) and the count of maxima ----
  unsigned long long s = 0ull;
  uint32_t cm = 0u;
  if (!bad) {
    const float2 mM = make_float2(-mc, -mc), cc = make_float2(c1, c1);
    uint32_t cm2 = 0u;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const uint4 v = sbuf[u * 32 + lane];
      float x[VE];
      Tr::values(v, x);
      float2 w2[VE / 2];
#pragma unroll
      for (int h = 0; h < VE / 2; ++h) {
        const float2 e = __fmul2_rn(__fadd2_rn(make_float2(x[2 * h], x[2 * h + 1]), mM), cc);
        w2[h] = make_float2(ex2_approx(e.x), ex2_approx(e.y));
      }
      float2 a;
      if constexpr (VE == 8) a = __fadd2_rn(__fadd2_rn(w2[0], w2[2]), __fadd2_rn(w2[1], w2[3]));
      else a = __fadd2_rn(w2[0], w2[1]);
      s += mass_fx(a.x + a.y);
      if constexpr (kHeadOnly) {
      } else if constexpr (VE == 8) {
        const __nv_bfloat162 M2 = __float2bfloat162_rn(mc);   // a bf16 value: exact
        cm2 += __heq2_mask(Tr::pair(v.x), M2) & 0x00010001u;
        cm2 += __heq2_mask(Tr::pair(v.y), M2) & 0x00010001u;
        cm2 += __heq2_mask(Tr::pair(v.z), M2) & 0x00010001u;
        cm2 += __heq2_mask(Tr::pair(v.w), M2) & 0x00010001u;
      } else {
#pragma unroll
        for (int i = 0; i < VE; ++i) cm += x[i] == mc ? 1u : 0u;
      }
    }
    cm += (cm2 & 0xFFFFu) + (cm2 >> 16);
  }
  s = warp_sum_u64(s);
  if (!kHeadOnly) cm = warp_sum_u32(cm);
  if (coded && !bad) piece_codes<T>(e_begin, k0, k1, rid, st_lo, st_hi, code_out);
  if (lane == 0) {
    uint4* o = reinterpret_cast<uint4*>(rec_out);
    o[0] = make_uint4(bad ? 0x7FC00000u : __float_as_uint(mc), timeout ? kTimeoutCnt : cm, (uint32_t)s, (uint32_t)(s >> 32));
    if (!kHeadOnly) o[1] = make_uint4(__float_as_uint(mn), 0u, 0u, 0u);
  }
}

// ------------------------------------------------------------------------------------------------
// The two kernels.
// ------------------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kStreamThreads, 3) piece_kernel(const Params p, const StreamWs ws, int np) {
  using Tr = Traits<T>;
  extern __shared__ __align__(128) unsigned char dyn[];
  PieceSmem& S = *reinterpret_cast<PieceSmem*>(dyn);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const long long total = (long long)p.B * np;
  const long long nw = (long long)gridDim.x * kItemPieces;
  const long long first = (long long)blockIdx.x * kItemPieces + warp;
  if (t < 2 * kItemPieces) mbar_init(&S.bar[t >> 1][t & 1], 1);
  fence_mbar_init();
  __syncthreads();   // the only CTA barrier: the mbarriers are initialised

  auto full_piece = [&](int pc) -> bool { return p.tma && (int64_t)(pc + 1) * kPieceElems<T> <= p.V; };
  int uses[2] = {0, 0};
  bool armed[2] = {false, false}, inflight[2] = {false, false};
  bool dead = false;   // a load wait ran out: no more bulk copies from this warp
  // the bulk copy of piece `it` (a full piece of an aligned row) into this warp's buffer b
  auto issue = [&](long long it, int b) {
    if (dead || it >= total) return;
    const int64_t row = it / np;
    const int pc = (int)(it - row * np);
    if (!full_piece(pc)) return;
    if (lane == 0) {
      fence_proxy_async_shared();
      mbar_arrive_expect_tx(&S.bar[warp][b], (uint32_t)kPieceBytes);
      if (!p.drop_loads)
        bulk_copy_g2s(&S.buf[warp][b][0], p.x + (row * p.ld + (int64_t)pc * kPieceElems<T>) * Tr::ESIZE,
                      (uint32_t)kPieceBytes, &S.bar[warp][b]);
    }
    armed[b] = true;
    inflight[b] = !p.drop_loads;
  };

  issue(first, 0);
  int k = 0;
  for (long long it = first; it < total; it += nw, ++k) {
    const int b = k & 1;
    __syncwarp();      // every lane has finished reading buffer b ^ 1 (the previous piece)
    issue(it + nw, b ^ 1);
    const int64_t row = it / np;
    const int pc = (int)(it - row * np);
    bool timeout = false;
    const uint4* sbuf = nullptr;
    if (armed[b]) {
      armed[b] = false;
      if (mbar_wait_bounded(&S.bar[warp][b], (uint32_t)(uses[b] & 1), p.wait_cycles)) {
        ++uses[b];
        inflight[b] = false;
        sbuf = &S.buf[warp][b][0];
      } else {
        timeout = true;
        dead = true;
      }
    }
    timeout = __any_sync(kFullMask, timeout);
    const float temp0 = p.temperature ? p.temperature[row] : 1.f;
    const float Teff = temp0 > 0.f ? temp0 : 1.f;
    const float invT = 1.f / Teff;
    const float c1 = kLog2e * invT;
    PieceRec* rec = ws.recs + row * ws.rec_ld + pc;
    const bool coded = row_coded(p, row);
    uint32_t k0 = 0u, k1 = 0u, rid = (uint32_t)row, st_lo = 0u, st_hi = 0u;
    if (coded) {
      const uint64_t sd = p.seed ? p.seed[row] : 0ull;
      const uint64_t stp = p.step ? p.step[row] : 0ull;
      k0 = (uint32_t)sd;
      k1 = (uint32_t)(sd >> 32);
      st_lo = (uint32_t)stp;
      st_hi = (uint32_t)(stp >> 32);
      if (p.row_id) rid = p.row_id[row];
    }
    // the Philox counters use the token's global index (a vocabulary shard starts at p.v0)
    if (sbuf) {
      piece_pass_full<T>(sbuf, p.v0 + (int64_t)pc * kPieceElems<T>, c1, timeout, coded, k0, k1, rid, st_lo, st_hi,
                         rec, ws.codes + (row * np + pc) * 32);
    } else {
      piece_stats_partial<T>(p.x + row * p.ld * Tr::ESIZE, p.V, p.tma, (int64_t)pc * kPieceElems<T>, c1, timeout, rec);
      if (coded && !timeout) piece_codes<T>(p.v0 + (int64_t)pc * kPieceElems<T>, k0, k1, rid, st_lo, st_hi,
                                            ws.codes + (row * np + pc) * 32);
    }
  }
  // a bulk copy of this warp that may still be landing (after a timed-out wait)
  for (int b2 = 0; b2 < 2; ++b2)
    if (inflight[b2]) (void)mbar_wait_bounded(&S.bar[warp][b2], (uint32_t)(uses[b2] & 1), 4000000000LL);
}

// One CTA per row (rows blockIdx.x, blockIdx.x + gridDim.x, ...).
template <typename T>
__global__ void __launch_bounds__(kStreamThreads) row_finish_kernel(const Params p, const StreamWs ws, int np) {
  __shared__ FinishSmem S;
  for (int64_t row = blockIdx.x; row < p.B; row += gridDim.x) {
    finish_row<T>(p, ws, row, np, S);
    __syncthreads();
  }
}

}  // namespace vsamp
