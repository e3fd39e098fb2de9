// The split-vocabulary sampling path: vsamp_sample with a caller-provided workspace.
//
// Every row is cut into fixed 64 KB chunks (32768 bf16 / 16384 fp32 logits); two streaming kernels sweep all
// (row, chunk) pairs of the batch with no per-row synchronisation inside a kernel:
//   split_stats_kernel  reads each chunk once from HBM and computes, in one pass, its maximum, its count of
//                       maxima and its mass sum(2^((x - m_c) * log2e / T)): every thread keeps a running
//                       maximum and a binary32 sum relative to it (rescaled when the maximum grows), and the
//                       threads' sums are rescaled to the chunk maximum m_c and added in 2^-40 fixed point.
//                       The last chunk of a row to finish (an atomic ticket) plans
//                       the row with the whole CTA: M = max m_c, S = sum of the chunk masses rescaled to M,
//                       the top-k / top-p / min-p cut (radix rounds and min-p statistics scan the row from
//                       L2 when the cut leaves the maximum's tie group), the cut's last kept index, and the
//                       draw's prune bound. Rows that keep one token get their outputs here.
//   split_draw_kernel   reads each chunk again (from L2) and draws: one Philox4x32-10 word per kept token, the
//                       prune bound, the exact perturbed score of the few candidates, and a 64-bit atomic
//                       maximum of (score, index) per row, published by every warp. The last warp of a row
//                       certifies the draw and writes the row's outputs.
// Chunking depends only on V, so results are deterministic and do not depend on the batch.
#pragma once

#include "vsamp_row.cuh"

namespace vsamp {

constexpr int kSplitThreads = 256;
constexpr int kChunkBytes = 65536;   // 256 threads x 16 vectors of 16 bytes
constexpr int kSplitVec = 16;        // vectors per thread

struct ChunkStat {                   // 16 bytes per (row, chunk)
  float m;                           // chunk maximum (NaN flags a non-finite value)
  uint32_t cnt;                      // elements equal to m
  unsigned long long s;              // sum of 2^((x - m) * c1), 2^-40 fixed point
};

struct RowPlan {                     // 128 bytes per row
  uint32_t done1, done2;             // chunks finished in each kernel (the last chunk resets its counter)
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
  uint32_t pad[7];
};
static_assert(sizeof(RowPlan) == 128, "RowPlan layout");
static_assert(sizeof(ChunkStat) == 16, "ChunkStat layout");

__host__ __device__ inline int64_t split_chunk_elems(int esize) { return kChunkBytes / esize; }
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
// The row planner: the last chunk's CTA of split_stats_kernel, once every chunk of the row is done.
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
#pragma unroll
        for (int i = 0; i < VE; ++i) x[i] = i < cnt ? Tr::load_global(xr, e + i) : -INFINITY;
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
  // -1 if there are fewer
  __device__ int32_t nth_equal(float xv, unsigned long long need, int64_t begin_vec) {
    int32_t found = -1;
    unsigned long long before = 0;
    for_each_tile(begin_vec, [&](int64_t, int64_t e, const float (&x)[VE], int cnt) {
      uint32_t c = 0;
#pragma unroll
      for (int i = 0; i < VE; ++i) c += (i < cnt && x[i] == xv) ? 1u : 0u;
      uint32_t tot;
      const uint32_t pre = block_scan_u32(c, tot, sh);
      const bool here = before + pre < need && need <= before + pre + c;
      if (here) {
        unsigned long long seen = before + pre;
#pragma unroll
        for (int i = 0; i < VE; ++i)
          if (i < cnt && x[i] == xv && ++seen == need) sh.i[0] = (int32_t)(e + i);
      }
      const bool done = before + tot >= need;
      before += tot;
      __syncthreads();
      if (done) found = sh.i[0];
      __syncthreads();
      return !done;
    });
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
    const float mk = stats[row * nchunks + k].m;
    if (mk != mk) nonfin = 1;
    else m = fmaxf(m, mk);
  }
  nonfin = __syncthreads_or(nonfin);
  const float M = block_max_f(m, sh);
  unsigned long long Sp = 0;
  uint32_t cMp = 0;
  for (int k = t; k < nchunks; k += kSplitThreads) {
    const ChunkStat cs = stats[row * nchunks + k];
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
  // the row's chunk statistics are zeroed once used and its counter reset, so that every completed call
  // leaves the workspace's counters and statistics zero whatever the next call's B and V
  auto finish = [&](int st, int draw) {
    __syncthreads();
    for (int k = t; k < nchunks; k += kSplitThreads) stats[row * nchunks + k] = ChunkStat{0.f, 0u, 0ull};
    if (t == 0) {
      pl.status = st;
      pl.draw = draw;
      pl.done1 = 0u;
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
    if (ck_mode == 1 || cp_mode == 1) path |= PATH_MAXGROUP;
    if (minp_on) {
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
        const ChunkStat cs = stats[row * nchunks + k];
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
    const unsigned long long skip = sh.bq[3];
    const int64_t begin_vec = cb * (split_chunk_elems(Tr::ESIZE) / VE);
    It = P.nth_equal(M, need - skip, begin_vec);
  } else {
    const unsigned long long need = fin.whole ? fin.cnt_eq : fin.need;
    It = P.nth_equal(xP, need, 0);
  }
  if (It < 0) {   // cannot happen with consistent counts; reported as an error
    write_outputs(-1, __int_as_float(0x7FC00000), VSAMP_ERR_INVALID_ARG, 0u);
    finish(VSAMP_ERR_INVALID_ARG, 0);
    return;
  }
  if (one_token) {
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
  }
  finish(VSAMP_OK, 1);
}

// ------------------------------------------------------------------------------------------------
// Kernel 1: chunk statistics in one pass; the last chunk of each row plans the row.
// ------------------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kSplitThreads) split_stats_kernel(const Params p, RowPlan* plans,
                                                                    ChunkStat* stats, int nchunks) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  __shared__ SplitShared sh;
  const int64_t row = p.row0 + blockIdx.y;
  const int64_t c = blockIdx.x;
  const int t = threadIdx.x;
  const float temp0 = p.temperature ? p.temperature[row] : 1.f;
  const float Teff = temp0 > 0.f ? temp0 : 1.f;   // greedy rows use T = 1 for their statistics
  const float c1 = kLog2e * (1.f / Teff);
  const unsigned char* xr = p.x + (int64_t)row * p.ld * Tr::ESIZE;
  const int64_t K = split_chunk_elems(Tr::ESIZE);

  // ---- one pass: running maximum m_t, binary32 mass relative to it, its count, non-finite check.
  // Vectors are loaded four at a time, the next four while the current ones are reduced. ----
  float m_t = -INFINITY, s_t = 0.f, nf = 0.f;
  uint32_t cnt_t = 0;
  const float2 cc = make_float2(c1, c1);
  auto vec = [&](const uint4& v, int cnt) {
    float x[VE];
    Tr::values(v, x);
    float vm = -INFINITY;
    if (cnt == VE) {
#pragma unroll
      for (int i = 0; i < VE; ++i) { vm = fmaxf(vm, x[i]); nf = fmaf(x[i], 0.f, nf); }
    } else {
#pragma unroll
      for (int i = 0; i < VE; ++i)
        if (i < cnt) { vm = fmaxf(vm, x[i]); nf = fmaf(x[i], 0.f, nf); }
    }
    if (vm > m_t) {
      s_t = m_t == -INFINITY ? 0.f : s_t * ex2_approx((m_t - vm) * c1);
      cnt_t = 0;
      m_t = vm;
    }
    float w[VE];
    if (cnt == VE) {
      const float2 mM = make_float2(-m_t, -m_t);
#pragma unroll
      for (int h = 0; h < VE / 2; ++h) {
        const float2 a = __fmul2_rn(__fadd2_rn(make_float2(x[2 * h], x[2 * h + 1]), mM), cc);
        w[2 * h] = ex2_approx(a.x);
        w[2 * h + 1] = ex2_approx(a.y);
      }
#pragma unroll
      for (int i = 0; i < VE; ++i) cnt_t += x[i] == m_t ? 1u : 0u;
    } else {
#pragma unroll
      for (int i = 0; i < VE; ++i) {
        const bool ok = i < cnt;
        const float d = x[i] - m_t;
        w[i] = ok ? ex2_approx(d * c1) : 0.f;
        cnt_t += (ok && d == 0.f) ? 1u : 0u;
      }
    }
#pragma unroll
    for (int h = VE / 2; h >= 1; h >>= 1)
#pragma unroll
      for (int i = 0; i < h; ++i) w[i] += w[i + h];
    s_t += w[0];
  };
  constexpr int kBatch = 4;
  const int64_t base = c * K + (int64_t)t * VE;
  uint4 cur[kBatch], nxt[kBatch];
  int ccnt[kBatch], ncnt[kBatch];
#pragma unroll
  for (int i = 0; i < kBatch; ++i) ccnt[i] = load_vec<T, false>(p, xr, base + (int64_t)i * kSplitThreads * VE, cur[i]);
#pragma unroll 1
  for (int j0 = 0; j0 < kSplitVec; j0 += kBatch) {
    if (j0 + kBatch < kSplitVec) {
#pragma unroll
      for (int i = 0; i < kBatch; ++i)
        ncnt[i] = load_vec<T, false>(p, xr, base + (int64_t)(j0 + kBatch + i) * kSplitThreads * VE, nxt[i]);
    }
#pragma unroll
    for (int i = 0; i < kBatch; ++i)
      if (ccnt[i]) vec(cur[i], ccnt[i]);
#pragma unroll
    for (int i = 0; i < kBatch; ++i) { cur[i] = nxt[i]; ccnt[i] = ncnt[i]; }
  }
  const uint32_t bad = __syncthreads_or(nf != 0.f ? 1 : 0);
  const float mc = block_max_f(m_t, sh);
  // the threads' masses rescaled to the chunk maximum, in 2^-40 fixed point (binary64 for the product)
  unsigned long long s = 0;
  uint32_t cm = 0;
  if (m_t == mc) {
    s = __double2ull_rn((double)s_t * 1099511627776.0);
    cm = cnt_t;
  } else if (m_t != -INFINITY) {
    s = __double2ull_rn((double)s_t * (double)ex2_approx((m_t - mc) * c1) * 1099511627776.0);
  }
  s = block_sum_u64(s, sh);
  cm = block_sum_u32(cm, sh);
  if (t == 0) {
    ChunkStat cs;
    cs.m = bad ? __int_as_float(0x7FC00000) : mc;
    cs.cnt = cm;
    cs.s = s;
    stats[row * nchunks + c] = cs;
    __threadfence();
    sh.ticket = atomicAdd(&plans[row].done1, 1u);
  }
  __syncthreads();
  if (sh.ticket != (uint32_t)(nchunks - 1)) return;
  __threadfence();
  plan_row<T>(p, plans, stats, stats, nchunks, row, temp0, Teff, c1, sh);
}

// ------------------------------------------------------------------------------------------------
// Kernel 2: the draw. Every chunk's best candidate meets the row's in a 64-bit atomic maximum; the last
// chunk certifies it and writes the outputs.
// ------------------------------------------------------------------------------------------------
template <typename T>
__global__ void __launch_bounds__(kSplitThreads) split_draw_kernel(const Params p, RowPlan* plans, int nchunks) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  constexpr int kWarps = kSplitThreads / 32;
  __shared__ uint4 splan[8];
  const int64_t row = p.row0 + blockIdx.y;
  const int t = threadIdx.x, lane = t & 31;
  RowPlan* gpl = plans + row;
  if (t < 8) splan[t] = reinterpret_cast<const uint4*>(gpl)[t];
  __syncthreads();
  const RowPlan& pl = *reinterpret_cast<const RowPlan*>(splan);
  if (pl.status != VSAMP_OK || !pl.draw) return;
  const float M = pl.M, xP = pl.xP;
  const int32_t It = pl.It;
  const uint32_t bk = pl.bk, rid = pl.rid, st_lo = pl.st_lo, st_hi = pl.st_hi;
  const bool all_cand = pl.all_cand != 0;
  const PhiloxKey key{pl.k0, pl.k1};

  // indices fit 32 bits (V < 2^31, checked on the host)
  const unsigned char* xr = p.x + (int64_t)row * p.ld * Tr::ESIZE;
  const int32_t n = (int32_t)p.V;
  const int32_t K = (int32_t)split_chunk_elems(Tr::ESIZE);
  const int32_t cbeg = (int32_t)blockIdx.x * K;
  const int32_t ebase = cbeg + t * VE;              // the thread's vector j starts at ebase + j * kStep
  constexpr int32_t kStep = kSplitThreads * VE;
  // kept: x > xP, or x == xP and index <= It; the groups of four tokens of a vector holding a kept token
  auto kept_groups = [&](const uint4& v, int32_t e0, int cnt) -> uint32_t {
    if (cnt == VE && e0 + VE - 1 <= It && Tr::all_ge(v, xP)) return (1u << (VE / 4)) - 1u;
    float x[VE];
    Tr::values(v, x);
    uint32_t gm = 0u;
#pragma unroll
    for (int i = 0; i < VE; ++i)
      if (i < cnt && (x[i] > xP || (x[i] == xP && e0 + i <= It))) gm |= 1u << (i >> 2);
    return gm;
  };
  const PhiloxRoundKeys rk(key);
  auto min_word = [&](int32_t e0, uint32_t gmask) -> uint32_t {
    uint32_t bmin = 0xFFFFFFFFu;
    const uint32_t g0 = (uint32_t)e0 >> 2;
#pragma unroll
    for (int g = 0; g < VE / 4; ++g) {
      if (!((gmask >> g) & 1u)) continue;
      const uint4 w4 = philox4x32_10_rk(make_uint4(g0 + (uint32_t)g, rid, st_lo, st_hi), rk);
      bmin = min(bmin, min(min(w4.x, w4.y), min(w4.z, w4.w)));
    }
    return bmin;
  };

  // ---- one Philox word per kept token; a vector is flagged when a kept token's word is below bk ----
  uint32_t flagged = 0;
  if (!all_cand && cbeg + K <= n && p.tma) {
    // a whole aligned chunk: 16-byte loads, four vectors in flight ahead of the ones being drawn
    const uint4* src = reinterpret_cast<const uint4*>(xr) + (ebase / VE);
    constexpr int kBatch = 4;
    uint4 cur[kBatch], nxt[kBatch];
#pragma unroll
    for (int i = 0; i < kBatch; ++i) cur[i] = __ldcs(src + i * kSplitThreads);
#pragma unroll 1
    for (int j0 = 0; j0 < kSplitVec; j0 += kBatch) {
      if (j0 + kBatch < kSplitVec) {
#pragma unroll
        for (int i = 0; i < kBatch; ++i) nxt[i] = __ldcs(src + (j0 + kBatch + i) * kSplitThreads);
      }
      // every vector of the batch lies at or before the cut's last index: only the values decide
      const bool below = ebase + (j0 + kBatch - 1) * kStep + VE - 1 <= It;
#pragma unroll 1
      for (int i = 0; i < kBatch; ++i) {
        const int32_t e0 = ebase + (j0 + i) * kStep;
        const uint32_t gm = (below && Tr::all_ge(cur[i], xP)) ? (1u << (VE / 4)) - 1u : kept_groups(cur[i], e0, VE);
        if (gm && min_word(e0, gm) < bk) flagged |= 1u << (j0 + i);
      }
#pragma unroll
      for (int i = 0; i < kBatch; ++i) cur[i] = nxt[i];
    }
  } else {
    for (int j = 0; j < kSplitVec; ++j) {
      const int32_t e0 = ebase + j * kStep;
      uint4 v;
      const int cnt = load_vec<T, true>(p, xr, e0, v);
      if (cnt == 0) break;
      const uint32_t gm = kept_groups(v, e0, cnt);
      if (!gm) continue;
      if (all_cand || min_word(e0, gm) < bk) flagged |= 1u << j;
    }
  }
  // ---- the flagged vectors' kept tokens: exact perturbed scores ----
  float bscore = -INFINITY;
  int32_t bidx = 0x7FFFFFFF;
  if (flagged) {
    const float invT = pl.invT, c1 = pl.c1, kappa = pl.kappa;
    while (flagged) {
      const int j = __ffs(flagged) - 1;
      flagged &= flagged - 1u;
      const int32_t e0 = ebase + j * kStep;
      uint4 v;
      const int cnt = load_vec<T, false>(p, xr, e0, v);
      float x[VE];
      Tr::values(v, x);
      uint32_t b[VE];
      const uint32_t g0 = (uint32_t)e0 >> 2;
#pragma unroll
      for (int g = 0; g < VE / 4; ++g) {
        const uint4 w4 = philox4x32_10(make_uint4(g0 + (uint32_t)g, rid, st_lo, st_hi), key);
        b[4 * g + 0] = w4.x; b[4 * g + 1] = w4.y; b[4 * g + 2] = w4.z; b[4 * g + 3] = w4.w;
      }
#pragma unroll
      for (int i = 0; i < VE; ++i) {
        if (!(i < cnt && (x[i] > xP || (x[i] == xP && e0 + i <= It)))) continue;
        if (!all_cand && b[i] >= bk) continue;
        const float d = x[i] - M;
        const float sv = d * invT;
        if (!all_cand) {
          const float w = ex2_approx(d * c1);
          const float u = fmaf((float)b[i], kTwoM32, kTwoM33);
          if (!(u < w * kappa * 1.00001f)) continue;
        }
        const float score = gumbel_score(sv, b[i]);
        const int32_t idx = e0 + i;
        if (argmax_better(score, idx, bscore, bidx)) { bscore = score; bidx = idx; }
      }
    }
  }
  // ---- each warp's best -> the row's 64-bit maximum; the last warp of the row finishes it ----
  const ArgMax a = warp_argmax(ArgMax{bscore, bidx, 0.f});
  uint32_t ticket = 0u;
  if (lane == 0) {
    if (a.idx != 0x7FFFFFFF) {
      const unsigned long long k = ((unsigned long long)score_key(a.score) << 32) | (0xFFFFFFFFu - (uint32_t)a.idx);
      atomicMax(&gpl->best, k);
    }
    __threadfence();
    ticket = atomicAdd(&gpl->done2, 1u);
  }
  ticket = __shfl_sync(kFullMask, ticket, 0);
  if (ticket != (uint32_t)(nchunks * kWarps - 1)) return;
  __threadfence();
  // ---- the last warp: certify, write the outputs, reset the row's draw state ----
  unsigned long long best = 0ull;
  if (lane == 0) best = atomicAdd(&gpl->best, 0ull);
  best = __shfl_sync(kFullMask, best, 0);
  const float gscore = best ? score_of_key((uint32_t)(best >> 32)) : -INFINITY;
  const int32_t gidx = best ? (int32_t)(0xFFFFFFFFu - (uint32_t)best) : -1;
  const float B0 = pl.B0;
  int32_t tok = gidx;
  int path = pl.path;
  if (!(all_cand || (best && gscore > B0 + 1e-4f * fmaxf(1.f, fabsf(B0))))) {
    // the prune bound did not certify the draw (probability ~1e-9): every kept token of the row, exactly
    path |= PATH_FALLBACK;
    const float invT = pl.invT;
    float fs = -INFINITY;
    int32_t fi = 0x7FFFFFFF;
    for (int32_t e = lane; e < n; e += 32) {
      const float xv = Tr::load_global(p.x, (int64_t)row * p.ld + e);
      if (!(xv > xP || (xv == xP && e <= It))) continue;
      const uint4 w4 = philox4x32_10(make_uint4((uint32_t)e >> 2, rid, st_lo, st_hi), key);
      const float score = gumbel_score((xv - M) * invT, philox_word(w4, (int)(e & 3)));
      if (argmax_better(score, e, fs, fi)) { fs = score; fi = e; }
    }
    tok = warp_argmax(ArgMax{fs, fi, 0.f}).idx;
  }
  if (lane == 0) {
    int st = VSAMP_OK;
    if (tok >= 0 && tok < n) {
      const float xt = Tr::load_global(p.x, (int64_t)row * p.ld + tok);
      p.token[row] = tok;
      if (p.logprob) p.logprob[row] = fminf((xt - M) * pl.invT - pl.logS, 0.f);
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
    gpl->best = 0ull;   // the workspace is left as it was found
    gpl->done2 = 0u;
  }
}

}  // namespace vsamp
