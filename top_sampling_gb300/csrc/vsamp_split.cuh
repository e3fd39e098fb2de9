// The split-vocabulary sampling path (vsamp_sample_ws): every row is cut into fixed pieces of 1024 logits and
// streaming kernels sweep all (row, piece) pairs of the batch (see the section "The streaming sampler" below).
// The cut into pieces depends only on V, so results are deterministic and do not depend on the batch.
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

constexpr int32_t kDeferIndex = -2;   // RowPlan::It: the draw kernel finds the cut's last kept index

struct RowPlan {                     // 128 bytes per row
  uint32_t done1, done2;             // reserved (zero)
  unsigned long long best;           // draw: (orderable score << 32) | (0xFFFFFFFF - index); 0 = none
  int32_t status;                    // the row's status; the draw kernel skips rows that are not VSAMP_OK
  int32_t draw;                      // 1: the draw kernel draws the token; 0: the outputs are written
  float M, invT, c1, xP, logS, B0, kappa;
  int32_t It;                        // kept: x > xP, or x == xP and index <= It
  uint32_t bk;
  int32_t all_cand;
  uint32_t rid, st_lo, st_hi, k0, k1;
  int32_t passes, rounds, path;
  uint32_t kept;
  int32_t cb;                        // It == kDeferIndex: the chunk holding the cut's last kept maximum,
  uint32_t cneed;                    //   which is the cneed-th maximum of that chunk (the draw finds it)
  int32_t one;                       // the cut keeps one token (the first maximum): no draw
  uint32_t pad[4];
};
static_assert(sizeof(RowPlan) == 128, "RowPlan layout");
static_assert(sizeof(ChunkStat) == 16, "ChunkStat layout");

__host__ __device__ inline int64_t split_chunk_elems(int esize) { return kPieceBytes / esize; }
__host__ __device__ inline int64_t split_nchunks(int64_t V, int esize) {
  const int64_t k = split_chunk_elems(esize);
  return (V + k - 1) / k;
}

// round(w * 2^40) for 0 <= w < 8 without a 64-bit conversion instruction: v = w * 2^40 < 2^43 is split into
// h (a multiple of 2^21, by rounding at that granularity) and l = v - h (exact, |l| <= 2^20); both are
// turned into integers by adding a power of two that places the unit in the last mantissa bit. The sum is
// round-to-nearest-even of v because h is even.
__device__ __forceinline__ unsigned long long mass_fx_split(float w) {
  const float v = w * kMassScale;
  const float big = 26388279066624.0f;          // 1.5 * 2^44: unit in the last place 2^21
  const float h = (v + big) - big;
  const float l = v - h;
  const uint32_t hi = __float_as_uint(fmaf(h, 4.76837158203125e-07f, 8388608.0f)) - 0x4B000000u;   // h / 2^21
  const int32_t lo = (int32_t)(__float_as_uint(l + 12582912.0f) - 0x4B400000u);                   // round(l)
  return ((unsigned long long)hi << 21) + (unsigned long long)(long long)lo;
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

  // radix search over the whole row (as the row engine's, with the row read from L2 by this CTA)
  __device__ RadixOut radix(bool mass_mode, unsigned long long goal, float goal_p, bool want_mass) {
    RadixOut out{};
    out.ok = 1;
    uint32_t prefix = 0;
    unsigned long long cnt_above = 0, mass_above = 0;
    const bool hist_mass = want_mass || mass_mode;
    const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
    for (int shift = Tr::KB - 8; shift >= 0; shift -= 8) {
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
          if ((rk & hmask) == (prefix & hmask)) {
            const uint32_t bin = (rk >> shift) & 255u;
            if (bin != run_bin) { flush(); run_bin = bin; run_cnt = 0; run_mass = 0; }
            ++run_cnt;
            if (hist_mass) run_mass += mass_fx_split(ex2_approx((x[i] - M) * c1));
          }
        }
        flush();
        return true;
      });
      ++passes;
      ++rounds;
      __syncthreads();
      if (mass_mode && goal_p >= 0.f && shift == Tr::KB - 8) {
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
      prefix |= sel << shift;
      cnt_above += ac;
      mass_above += am;
      if (mass_mode) goal -= am; else goal -= ac;
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
  __device__ void minp_stats(uint32_t kmin32, uint32_t& cnt_ge, unsigned long long& mass_ge, uint32_t& minkey,
                             uint32_t& cnt_minkey) {
    uint32_t c = 0, mk = 0xFFFFFFFFu, cmk = 0;
    unsigned long long m = 0;
    for_each_tile(0, [&](int64_t, int64_t, const float (&x)[VE], int cnt) {
#pragma unroll
      for (int i = 0; i < VE; ++i) {
        const uint32_t k32 = key_f32_bits(__float_as_uint(x[i]));
        if (i < cnt && k32 >= kmin32) {
          ++c;
          m += mass_fx_split(ex2_approx((x[i] - M) * c1));
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
  __device__ int32_t nth_equal(float xv, unsigned long long need, int64_t begin_vec) {
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

// ------------------------------------------------------------------------------------------------
// The row's plan, by the CTA of its last chunk (out of line: the chunk pass keeps its registers).
// ------------------------------------------------------------------------------------------------
template <typename T>
static __device__ __noinline__ void plan_row(const Params p, RowPlan* plans, const ChunkStat* stats_c,
                                            ChunkStat* stats, int nchunks, int64_t row, float temp0, float Teff,
                                            float c1, SplitShared& sh) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  const int t = threadIdx.x;
  (void)stats_c;
  RowPlan& pl = plans[row];
  const int64_t n = p.V;
  // ---- combine the chunks: M, non-finite flag, S rescaled to M, count of maxima ----
  float m = -INFINITY;
  uint32_t nonfin = 0;
  for (int k = t; k < nchunks; k += kSplitThreads) {
    const float mk = load_stat(stats + row * nchunks + k).m;
    if (mk != mk) nonfin = 1;
    else m = fmaxf(m, mk);
  }
  nonfin = __syncthreads_or(nonfin);
  const float M = block_max_f(m, sh);
  unsigned long long Sp = 0;
  uint32_t cMp = 0;
  for (int k = t; k < nchunks; k += kSplitThreads) {
    const ChunkStat cs = load_stat(stats + row * nchunks + k);
    if (cs.m == M) {
      Sp += cs.s;
      cMp += cs.cnt;
    } else if (!nonfin) {
      // 2^((m_c - M) * c1) is below 1: the chunk's fixed-point mass rescaled in binary64
      const double f = exp2((double)((cs.m - M) * c1));
      Sp += (unsigned long long)__double2ull_rn((double)cs.s * f);
    }
  }
  const unsigned long long Sfx = block_sum_u64(Sp, sh);
  const uint32_t cM = block_sum_u32(cMp, sh);

  // ---- status ----
  float topp = p.top_p ? p.top_p[row] : 1.f;
  float minp = p.min_p ? p.min_p[row] : 0.f;
  const int32_t topk = p.top_k ? p.top_k[row] : 0;
  int status = VSAMP_OK;
  if (nonfin) status = VSAMP_ERR_NONFINITE;
  else if (isnan(temp0) || isinf(temp0) || isnan(topp) || !(topp > 0.f) || isnan(minp) || minp > 1.f)
    status = VSAMP_ERR_INVALID_ARG;
  const bool greedy = !(temp0 > 0.f);
  const float invT = 1.f / Teff;
  int path = p.tma ? 0 : PATH_NOTMA;
  RowPlanner<T> P{p, sh, row, n, M, c1};
  P.passes = 2;
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
  // the row's status, whether the draw kernel draws it, and its draw slot (the atomic maximum) cleared
  auto finish = [&](int st, int draw) {
    __syncthreads();
    if (t == 0) {
      pl.status = st;
      pl.draw = draw;
      pl.done1 = 0u;
      pl.done2 = 0u;
      pl.best = 0ull;
    }
  };
  if (status != VSAMP_OK) {
    write_outputs(-1, __int_as_float(0x7FC00000), status, 0u);
    finish(status, 0);
    return;
  }
  const float logS = logf(u64_to_float(Sfx) * 9.094947017729282379e-13f);   // 2^-40
  const unsigned long long one = 1ull << kMassShift;
  const uint32_t rkM = Tr::rkey_of_value(M);

  // ---- plan: the shortest prefix over top-k, top-p and min-p ----
  int plan_status = VSAMP_OK;
  Cut fin{};
  const bool minp_on = !greedy && minp > 0.f;
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
      uint32_t cnt_ge, minkey, cnt_minkey;
      unsigned long long mass_ge;
      P.minp_stats(key_f32_bits(__float_as_uint(xf)), cnt_ge, mass_ge, minkey, cnt_minkey);
      const uint32_t rkm = (Tr::KB == 32) ? minkey : (minkey >> 16);
      fin = Cut{rkm, (unsigned long long)(cnt_ge - cnt_minkey), cnt_minkey, cnt_minkey, mass_ge, 1};
    } else {
      fin = Cut{rkM, 0, (unsigned long long)n, 0, Sfx, 1};
    }
    if (ck_mode == 2) {
      const RadixOut r = P.radix(false, ck.need, -1.f, cp_mode == 2);
      if (!r.ok) plan_status = VSAMP_ERR_INVALID_ARG;
      const unsigned long long need = ck.need - r.cnt_above;
      const unsigned long long wP = mass_fx_split(ex2_approx((Tr::value_of_rkey(r.rk) - M) * c1));
      ck = Cut{r.rk, r.cnt_above, need, r.cnt_eq, r.mass_above + need * wP, 0};
      path |= PATH_RADIX_K;
      if (cp_mode == 2) cp_goal = ceil_mul_frac(topp, ck.mass);
    }
    if (cp_mode == 2 && plan_status == VSAMP_OK) {
      const RadixOut r = P.radix(true, cp_goal, goal_p, true);
      if (!r.ok) plan_status = VSAMP_ERR_INVALID_ARG;
      const unsigned long long wP = mass_fx_split(ex2_approx((Tr::value_of_rkey(r.rk) - M) * c1));
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
  if (plan_status != VSAMP_OK) {
    write_outputs(-1, __int_as_float(0x7FC00000), plan_status, 0u);
    finish(plan_status, 0);
    return;
  }

  // ---- the cut's last kept index ----
  const unsigned long long kept = fin.kept();
  const bool one_token = greedy || kept == 1;
  float xP = Tr::value_of_rkey(fin.rk);
  int32_t It = kAllIndex;
  int32_t cb_def = -1;
  uint32_t cneed_def = 0u;
  if (fin.whole && !one_token) {
    if (fin.above == 0 && fin.cnt_eq == 0) xP = -INFINITY;   // every element
  } else if (fin.rk == rkM) {
    // the need-th maximum: find its chunk from the chunk counts, then scan that chunk
    const unsigned long long need = fin.whole ? cM : fin.need;
    unsigned long long before = 0;
    int64_t cb = -1;
    for (int64_t k0 = 0; k0 < nchunks && cb < 0; k0 += kSplitThreads) {
      const int64_t k = k0 + t;
      uint32_t ck = 0;
      if (k < nchunks) {
        const ChunkStat cs = load_stat(stats + row * nchunks + k);
        ck = cs.m == M ? cs.cnt : 0u;
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
    // the draw kernel finds it in chunk cb, which it holds in shared memory anyway
    cb_def = (int32_t)cb;
    cneed_def = (uint32_t)(need - sh.bq[3]);
    It = kDeferIndex;
  } else {
    const unsigned long long need = fin.whole ? fin.cnt_eq : fin.need;
    It = P.nth_equal(xP, need, 0);
  }
  if (It < 0 && It != kDeferIndex) {   // cannot happen with consistent counts; reported as an error
    write_outputs(-1, __int_as_float(0x7FC00000), VSAMP_ERR_INVALID_ARG, 0u);
    finish(VSAMP_ERR_INVALID_ARG, 0);
    return;
  }
  if (one_token && It != kDeferIndex) {
    // the first maximum; (x - M) / T = 0
    write_outputs(It, fminf(-logS, 0.f), VSAMP_OK, (uint32_t)kept);
    finish(VSAMP_OK, 0);
    return;
  }
  // ---- the draw's prune bound: a token can beat B0 = ln(S_kept) - 3 only if u < w * kappa ----
  const float skept = fmaxf(u64_to_float(fin.mass) * 9.094947017729282379e-13f, 1.f);
  const float kappa = 20.085536923187668f / skept;
  const bool all_cand = kappa >= 0.99f;
  if (t == 0) {
    const uint64_t sd = p.seed ? p.seed[row] : 0ull;
    const uint64_t st = p.step ? p.step[row] : 0ull;
    pl.M = M;
    pl.invT = invT;
    pl.c1 = c1;
    pl.xP = xP;
    pl.It = It;
    pl.logS = logS;
    pl.kappa = kappa;
    pl.all_cand = all_cand ? 1 : 0;
    pl.bk = all_cand ? 0xFFFFFFFFu : __float2uint_ru(kappa * 1.00001f * 4294967296.0f);
    pl.B0 = -logf(kappa);
    pl.rid = p.row_id ? p.row_id[row] : (uint32_t)row;
    pl.st_lo = (uint32_t)st;
    pl.st_hi = (uint32_t)(st >> 32);
    pl.k0 = (uint32_t)sd;
    pl.k1 = (uint32_t)(sd >> 32);
    pl.passes = P.passes + 1;
    pl.rounds = P.rounds;
    pl.path = path;
    pl.kept = (uint32_t)kept;
    pl.cb = cb_def;
    pl.cneed = cneed_def;
    pl.one = one_token ? 1 : 0;
  }
  finish(VSAMP_OK, 1);
}

// ------------------------------------------------------------------------------------------------
// The streaming sampler: four kernels, ordered by the stream.
//   warp_stats_kernel    every warp independently takes 4 KB pieces of consecutive logits (grid-stride
//                        over (row, piece) items; lane l holds vectors u * 32 + l of the piece): the piece's
//                        maximum m_p, count of maxima and mass relative to m_p in 2^-40 fixed point summed per
//                        16-byte vector, read once from HBM.
//   stream_plan_kernel   one CTA per row: the row's plan from its piece statistics (radix rounds over the row
//                        only when the cut leaves the maximum's tie group).
//   warp_draw_kernel     the same items, each piece read again (mostly from L2): one Philox4x32-10 word per
//                        kept token, the prune bound, exact scores of the few candidates; a warp with a
//                        candidate meets the row's best in a 64-bit atomic maximum.
//   stream_finish_kernel one CTA per row: certify the draw and write the outputs.
// No warp waits for another inside a kernel, and the streaming kernels use no shared memory or CTA barriers.
// ------------------------------------------------------------------------------------------------
struct StreamHeader {       // the first 256 bytes of the workspace (reserved, left zero)
  uint32_t reserved[64];
};
static_assert(sizeof(StreamHeader) == 256, "StreamHeader layout");

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

// Statistics of every piece: one warp per item, grid-stride.
template <typename T>
__global__ void __launch_bounds__(kStreamThreads) warp_stats_kernel(const Params p, ChunkStat* stats, int np) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  constexpr int U = kPieceVecs<T>;
  const int lane = threadIdx.x & 31;
  const long long total = (long long)p.B * np;
  const long long nw = (long long)gridDim.x * (kStreamThreads / 32);
  for (long long it = (long long)blockIdx.x * (kStreamThreads / 32) + (threadIdx.x >> 5); it < total; it += nw) {
    const int64_t row = it / np;
    const int pc = (int)(it - row * np);
    const float temp0 = p.temperature ? p.temperature[row] : 1.f;
    const float Teff = temp0 > 0.f ? temp0 : 1.f;   // greedy rows use T = 1 for their statistics
    const float c1 = kLog2e * (1.f / Teff);
    const PieceView<T> pv{p.x + row * p.ld * Tr::ESIZE, p.V, p.tma, (int64_t)pc * kPieceElems<T>};
    if (it + nw < total) {
      const int64_t r2 = (it + nw) / np;
      const int pc2 = (int)(it + nw - r2 * np);
      PieceView<T>{p.x + r2 * p.ld * Tr::ESIZE, p.V, p.tma, (int64_t)pc2 * kPieceElems<T>}.prefetch();
    }
    uint4 v[U];
    int cnt[U];
    if (pv.full()) {
#pragma unroll
      for (int u = 0; u < U; ++u) { pv.get_full(u, v[u]); cnt[u] = VE; }
    } else {
#pragma unroll
      for (int u = 0; u < U; ++u) cnt[u] = pv.get(u, v[u]);
    }
    // ---- maximum and non-finite check ----
    float mt = -INFINITY, nf = 0.f;
#pragma unroll
    for (int u = 0; u < U; ++u) {
      float x[VE];
      Tr::values(v[u], x);
#pragma unroll
      for (int i = 0; i < VE; ++i)
        if (i < cnt[u]) { mt = fmaxf(mt, x[i]); nf = fmaf(x[i], 0.f, nf); }
    }
    const float mc = warp_max_f(mt);
    const bool bad = __any_sync(kFullMask, nf != 0.f);
    // ---- mass relative to the piece maximum (2^-40 fixed point per vector) and the count of maxima ----
    unsigned long long s = 0ull;
    uint32_t cm = 0u;
    if (!bad) {
      const float2 mM = make_float2(-mc, -mc), cc = make_float2(c1, c1);
#pragma unroll
      for (int u = 0; u < U; ++u) {
        float x[VE];
        Tr::values(v[u], x);
        if (cnt[u] == VE) {
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
        } else if (cnt[u] > 0) {
          float w[VE];
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
      ChunkStat cs;
      cs.m = bad ? __int_as_float(0x7FC00000) : mc;
      cs.cnt = cm;
      cs.s = s;
      stats[it] = cs;
    }
  }
}

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

// Exact perturbed scores of one vector's kept tokens that pass the prune bound (every kept token when the
// plan makes all of them candidates); the running arg-max is updated in place.
template <typename T>
__device__ __noinline__ void draw_exact(uint4 v, int cnt, int64_t e0, const RowPlan* plp, int32_t It, float& bscore,
                                        int32_t& bidx) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  const RowPlan& pl = *plp;
  const bool all_cand = pl.all_cand != 0;
  const PhiloxKey key{pl.k0, pl.k1};
  float x[VE];
  Tr::values(v, x);
  uint32_t b[VE];
#pragma unroll
  for (int g = 0; g < VE / 4; ++g) {
    const uint4 w4 = philox4x32_10(make_uint4((uint32_t)(e0 >> 2) + (uint32_t)g, pl.rid, pl.st_lo, pl.st_hi), key);
    b[4 * g + 0] = w4.x; b[4 * g + 1] = w4.y; b[4 * g + 2] = w4.z; b[4 * g + 3] = w4.w;
  }
#pragma unroll
  for (int i = 0; i < VE; ++i) {
    if (!(i < cnt && (x[i] > pl.xP || (x[i] == pl.xP && e0 + i <= (int64_t)It)))) continue;
    if (!all_cand && b[i] >= pl.bk) continue;
    const float d = x[i] - pl.M;
    const float sv = d * pl.invT;
    if (!all_cand) {
      const float w = ex2_approx(d * pl.c1);
      const float u = fmaf((float)b[i], kTwoM32, kTwoM33);
      if (!(u < w * pl.kappa * 1.00001f)) continue;
    }
    const float score = gumbel_score(sv, b[i]);
    const int32_t idx = (int32_t)(e0 + i);
    if (argmax_better(score, idx, bscore, bidx)) { bscore = score; bidx = idx; }
  }
}

// stream_finish_kernel: one CTA per row certifies the draw, writes the outputs and resets the row's draw
// slot. Rows whose plan does not draw were finished by the planner.
template <typename T>
__global__ void __launch_bounds__(kSplitThreads) stream_finish_kernel(const Params p, RowPlan* plans) {
  using Tr = Traits<T>;
  __shared__ uint4 fplan[8];
  __shared__ float bs[8];
  __shared__ int32_t bi[8];
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t row = blockIdx.x;
  RowPlan* gpl = plans + row;
  if (t < 8) fplan[t] = reinterpret_cast<const uint4*>(gpl)[t];
  __syncthreads();
  const RowPlan& pl = *reinterpret_cast<const RowPlan*>(fplan);
  if (pl.status == VSAMP_OK && pl.draw) {
    const unsigned long long best = pl.best;
    const float gscore = best ? score_of_key((uint32_t)(best >> 32)) : -INFINITY;
    int32_t tok = best ? (int32_t)(0xFFFFFFFFu - (uint32_t)best) : -1;
    int path = pl.path;
    const bool all_cand = pl.all_cand != 0;
    const float B0 = pl.B0;
    if (!pl.one && !(all_cand || (best && gscore > B0 + 1e-4f * fmaxf(1.f, fabsf(B0))))) {
      // the prune bound did not certify the draw (probability ~1e-9): every kept token of the row, exactly
      path |= PATH_FALLBACK;
      const PhiloxKey key{pl.k0, pl.k1};
      const float xP = pl.xP, M = pl.M, invT = pl.invT;
      const int32_t It = pl.It;
      float fs = -INFINITY;
      int32_t fi = 0x7FFFFFFF;
      for (int64_t e = t; e < p.V; e += kSplitThreads) {
        const float xv = Tr::load_global(p.x, row * p.ld + e);
        if (!(xv > xP || (xv == xP && e <= (int64_t)It))) continue;
        const uint4 w4 = philox4x32_10(make_uint4((uint32_t)(e >> 2), pl.rid, pl.st_lo, pl.st_hi), key);
        const float score = gumbel_score((xv - M) * invT, philox_word(w4, (int)(e & 3)));
        if (argmax_better(score, (int32_t)e, fs, fi)) { fs = score; fi = (int32_t)e; }
      }
      const ArgMax a = warp_argmax(ArgMax{fs, fi, 0.f});
      if (lane == 0) { bs[warp] = a.score; bi[warp] = a.idx; }
      __syncthreads();
      ArgMax b{bs[0], bi[0], 0.f};
      for (int w = 1; w < kSplitThreads / 32; ++w)
        if (argmax_better(bs[w], bi[w], b.score, b.idx)) b = ArgMax{bs[w], bi[w], 0.f};
      tok = b.idx;
    }
    if (t == 0) {
      int st = VSAMP_OK;
      if (tok >= 0 && (int64_t)tok < p.V) {
        const float xt = Tr::load_global(p.x, row * p.ld + tok);
        p.token[row] = tok;
        if (p.logprob) p.logprob[row] = pl.one ? fminf(-pl.logS, 0.f) : fminf((xt - pl.M) * pl.invT - pl.logS, 0.f);
      } else {
        st = VSAMP_ERR_INVALID_ARG;
        p.token[row] = -1;
        if (p.logprob) p.logprob[row] = __int_as_float(0x7FC00000);
      }
      if (p.row_status) p.row_status[row] = st;
      if (p.stats) {
        p.stats[row * 4 + 0] = pl.passes;
        p.stats[row * 4 + 1] = pl.rounds;
        p.stats[row * 4 + 2] = (int32_t)pl.kept;
        p.stats[row * 4 + 3] = path;
      }
    }
  }
  if (t == 0) gpl->best = 0ull;   // the draw slot is left zero
}

// One CTA per row: the row's plan from its chunk statistics.
template <typename T>
__global__ void __launch_bounds__(kSplitThreads) stream_plan_kernel(const Params p, RowPlan* plans, ChunkStat* stats,
                                                                   int nc) {
  __shared__ SplitShared sh;
  const int64_t r = blockIdx.x;
  const float temp0 = p.temperature ? p.temperature[r] : 1.f;
  const float Teff = temp0 > 0.f ? temp0 : 1.f;
  plan_row<T>(p, plans, stats, stats, nc, r, temp0, Teff, kLog2e * (1.f / Teff), sh);
}


// The draw over every piece of the rows whose plan draws: one warp per item of kDrawRun consecutive pieces of
// a row, grid-stride.
template <typename T>
__global__ void __launch_bounds__(kStreamThreads, 2) warp_draw_kernel(const Params p, RowPlan* plans, int np) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  constexpr int U = kPieceVecs<T>;
  constexpr int G = VE / 4;          // groups of four tokens (one Philox counter) per vector
  constexpr int NG = U * G;          // groups per lane and piece
  const int lane = threadIdx.x & 31;
  const int nruns = (np + kDrawRun - 1) / kDrawRun;
  const long long total = (long long)p.B * nruns;
  const long long nw = (long long)gridDim.x * (kStreamThreads / 32);
  for (long long it = (long long)blockIdx.x * (kStreamThreads / 32) + (threadIdx.x >> 5); it < total; it += nw) {
    const int64_t row = it / nruns;
    const int run = (int)(it - row * nruns);
    RowPlan* gp = plans + row;
    if (!(__ldg(&gp->status) == VSAMP_OK && __ldg(&gp->draw))) continue;
    const float xP = __ldg(&gp->xP);
    const int32_t It0 = __ldg(&gp->It);
    const int32_t cbp = __ldg(&gp->cb);
    const bool one = __ldg(&gp->one) != 0;
    const uint32_t bk = __ldg(&gp->bk);
    const bool all_cand = __ldg(&gp->all_cand) != 0;
    const PhiloxRowMin ph(PhiloxKey{__ldg(&gp->k0), __ldg(&gp->k1)}, __ldg(&gp->rid), __ldg(&gp->st_lo),
                          __ldg(&gp->st_hi));
    if (it + nw < total) {
      const int64_t r2 = (it + nw) / nruns;
      const int run2 = (int)(it + nw - r2 * nruns);
      for (int k = 0; k < kDrawRun && run2 * kDrawRun + k < np; ++k)
        PieceView<T>{p.x + r2 * p.ld * Tr::ESIZE, p.V, p.tma, (int64_t)(run2 * kDrawRun + k) * kPieceElems<T>}.prefetch();
    }
    float bscore = -INFINITY;
    int32_t bidx = 0x7FFFFFFF;
    bool cand = false;   // warp-uniform: some lane evaluated a candidate
#pragma unroll 1
    for (int k = 0; k < kDrawRun; ++k) {
      const int pc = run * kDrawRun + k;
      if (pc >= np) break;
      const PieceView<T> pv{p.x + row * p.ld * Tr::ESIZE, p.V, p.tma, (int64_t)pc * kPieceElems<T>};
      // the cut's last kept index: inside the maximum's tie group it lies in piece cb, found here
      int32_t It = It0;
      if (It == kDeferIndex)
        It = pc < cbp ? kAllIndex : (pc > cbp ? kNoIndex : piece_nth_equal<T>(pv, xP, __ldg(&gp->cneed)));
      if (one) {
        // one token is kept: the piece holding it publishes it (score +inf)
        if (pc == cbp && lane == 0 && It >= 0)
          atomicMax(&gp->best, ((unsigned long long)score_key(INFINITY) << 32) | (0xFFFFFFFFu - (uint32_t)It));
        continue;
      }
      uint32_t gmask = 0u;   // kept groups: bit u * G + g
      {
        uint4 v[U];
        int cnt[U];
        if (pv.full()) {
#pragma unroll
          for (int u = 0; u < U; ++u) { pv.get_full(u, v[u]); cnt[u] = VE; }
        } else {
#pragma unroll
          for (int u = 0; u < U; ++u) cnt[u] = pv.get(u, v[u]);
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int64_t e0 = pv.elem(u);
          if (cnt[u] == VE && e0 + VE - 1 <= (int64_t)It && Tr::all_ge(v[u], xP)) {
            gmask |= ((1u << G) - 1u) << (u * G);
          } else if (cnt[u] > 0) {
            float x[VE];
            Tr::values(v[u], x);
#pragma unroll
            for (int i = 0; i < VE; ++i)
              if (i < cnt[u] && (x[i] > xP || (x[i] == xP && e0 + i <= (int64_t)It))) gmask |= 1u << (u * G + (i >> 2));
          }
        }
      }
      // ---- one Philox word per kept token; a vector is flagged when a kept token's word is below bk ----
      uint32_t flagged = 0u;
      if (all_cand) {
#pragma unroll
        for (int u = 0; u < U; ++u)
          if ((gmask >> (u * G)) & ((1u << G) - 1u)) flagged |= 1u << u;
      } else if (gmask) {
        // counter word of group gi = u * G + g: (first element of vector u) / 4 + g
        const uint32_t cb0 = (uint32_t)(pv.elem(0) >> 2);
        auto ctr = [&](int gi) -> uint32_t { return cb0 + (uint32_t)((gi / G) * 32 * G + gi % G); };
        if (gmask == (uint32_t)((1ull << NG) - 1ull)) {
          // every token of the lane's vectors is kept: four counters at a time
#pragma unroll 1
          for (int g0 = 0; g0 < NG; g0 += 4) {
            const uint32_t c4[4] = {ctr(g0), ctr(g0 + 1), ctr(g0 + 2), ctr(g0 + 3)};
            uint32_t m[4];
            ph.min_words<4>(c4, m);
#pragma unroll
            for (int q = 0; q < 4; ++q)
              if (m[q] < bk) flagged |= 1u << ((g0 + q) / G);
          }
        } else {
#pragma unroll 1
          for (int gi = 0; gi < NG; ++gi) {
            if (!((gmask >> gi) & 1u)) continue;
            const uint32_t c1[1] = {ctr(gi)};
            uint32_t m[1];
            ph.min_words<1>(c1, m);
            if (m[0] < bk) flagged |= 1u << (gi / G);
          }
        }
      }
      // ---- flagged vectors (rare): exact perturbed scores ----
      if (__any_sync(kFullMask, flagged != 0u)) {
        cand = true;
        while (flagged) {
          const int u = __ffs(flagged) - 1;
          flagged &= flagged - 1u;
          uint4 v;
          const int cnt = pv.get(u, v);
          draw_exact<T>(v, cnt, pv.elem(u), gp, It, bscore, bidx);
        }
      }
    }
    // ---- the warp's best meets the row's ----
    if (cand) {
      const ArgMax a = warp_argmax(ArgMax{bscore, bidx, 0.f});
      if (lane == 0 && a.idx != 0x7FFFFFFF)
        atomicMax(&gp->best, ((unsigned long long)score_key(a.score) << 32) | (0xFFFFFFFFu - (uint32_t)a.idx));
    }
  }
}

}  // namespace vsamp
