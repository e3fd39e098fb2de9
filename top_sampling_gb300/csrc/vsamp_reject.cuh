// The dual-pivot rejection sampler (vsamp_sample_rejection): a draw from the filtered distribution without a sort
// or a radix cut ("Sorting-free top-k/top-p/min-p sampling with dual-pivot rejection kernels #901", Background:
// top-k, top-p, min-p and joint rounds over a shrinking interval; Task: a cap on the rounds, a fallback to the
// exact cut on overflow, counted; one batch-wide launch with per-row parameters).
//
// One CTA per row, the row read from global memory (mostly L2) at every pass. Masses are 2^-40 fixed-point integers
// per element, so every prefix sum is exact and the candidate a scan flags does not depend on the launch. Per row:
//   pass 0   the maximum M, the fixed-point mass S of w = exp((x - M) / T), the count of maxima, non-finite check.
//   rounds   the proposal set is a prefix of the order (value desc, index asc), {x > lx} u {x == lx, index < li};
//            each round draws a uniform u from Philox4x32-10 (counter (2^32 - 1 - round, row_id, step), word 0),
//            scans the set's fixed-point CDF in index order for the candidate c where it first exceeds u times the
//            set's mass (pivot_0 = x_c), and counts, in one pass, the tokens and mass above pivot_0 and above
//            pivot_1 = (pivot_0 + high) / 2 and the tokens equal to pivot_0 before c. c is accepted iff its rank
//            in the order is inside the kept prefix: rank < k (top-k), prefix mass before c < p * S_k (top-p on the
//            top-k mass S_k, counted once by a radix count search when both are on), w_c >= min_p (min-p). A
//            rejected c moves the set's end to c (everything after it in the order is outside too); if everything
//            at or below pivot_1 is outside as well, the set ends above pivot_1, else high = pivot_1.
//   cap      after 32 rounds the row takes the exact cut (radix rounds) and one CDF draw inside it
//            (PATH_REJECT_CAP in stats).
// Accepting exactly the candidates inside the kept prefix, from proposals proportional to w on a superset of it,
// gives a draw proportional to w on the kept prefix: the same law as vsamp_sample, from other random numbers.
#pragma once

#include "vsamp_host.h"
#include "vsamp_split.cuh"

namespace vsamp {

enum : int { PATH_REJECT_CAP = 64 };   // stats[r][3]: the rejection rounds hit their cap; drawn from the exact cut
constexpr int kRejectRounds = 32;

__device__ __forceinline__ unsigned long long elem_mass(float x, float M, float c1) {
  return mass_fx(ex2_approx((x - M) * c1));
}
// inside the proposal set {x > lx} u {x == lx, i < li}
__device__ __forceinline__ bool in_set(float x, int64_t i, float lx, int64_t li) {
  return x > lx || (x == lx && i < li);
}

// exclusive prefix of v over the CTA's threads in index order, and the block total (64-bit)
__device__ __forceinline__ unsigned long long block_scan_u64(unsigned long long v, unsigned long long& total,
                                                             SplitShared& sh) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  unsigned long long incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const unsigned long long y = __shfl_up_sync(kFullMask, incl, o);
    if (lane >= o) incl += y;
  }
  __syncthreads();
  if (lane == 31) sh.q[warp][1] = incl;
  __syncthreads();
  unsigned long long base = 0, tot = 0;
#pragma unroll
  for (int w = 0; w < kSplitThreads / 32; ++w) {
    const unsigned long long x = sh.q[w][1];
    if (w < warp) base += x;
    tot += x;
  }
  total = tot;
  return base + incl - v;
}

template <typename T>
struct RejectRow {
  using Tr = Traits<T>;
  static constexpr int VE = Tr::VE;
  const Params& p;
  SplitShared& sh;
  int64_t row, n;
  float M, c1;

  __device__ __forceinline__ int load(int64_t vi, float (&x)[VE]) const {
    const unsigned char* xr = p.x + row * p.ld * Tr::ESIZE;
    uint4 v;
    const int cnt = load_vec<T, false>(p, xr, vi * VE, v);
    Tr::values(v, x);
    return cnt;
  }

  // the first index (index order) where the fixed-point CDF of the set {x > lx} u {x == lx, i < li} exceeds
  // `target` (0 <= target < the set's mass); -1 if it never does
  __device__ __noinline__ int32_t cdf_pick(float lx, int64_t li, unsigned long long target) {
    const int64_t nvec = (n + VE - 1) / VE;
    unsigned long long before = 0;
    int32_t found = -1;
    for (int64_t v0 = 0; v0 < nvec; v0 += kSplitThreads) {
      const int64_t vi = v0 + threadIdx.x;
      float x[VE];
      int cnt = 0;
      unsigned long long mine = 0;
      if (vi < nvec) {
        cnt = load(vi, x);
#pragma unroll
        for (int i = 0; i < VE; ++i)
          if (i < cnt && in_set(x[i], vi * VE + i, lx, li)) mine += elem_mass(x[i], M, c1);
      }
      unsigned long long tot;
      const unsigned long long excl = block_scan_u64(mine, tot, sh);
      if (mine && before + excl <= target && target < before + excl + mine) {
        unsigned long long run = before + excl;
#pragma unroll
        for (int i = 0; i < VE; ++i) {
          if (i < cnt && in_set(x[i], vi * VE + i, lx, li)) {
            run += elem_mass(x[i], M, c1);
            if (target < run) { sh.i[0] = (int32_t)(vi * VE + i); break; }
          }
        }
      }
      const bool done = target < before + tot;
      before += tot;
      __syncthreads();
      if (done) { found = sh.i[0]; break; }
      __syncthreads();
    }
    return found;
  }

  // fixed-point mass of the set {x > lx} u {x == lx, i < li}
  __device__ __noinline__ unsigned long long set_mass(float lx, int64_t li) {
    const int64_t nvec = (n + VE - 1) / VE;
    unsigned long long m = 0;
    for (int64_t vi = threadIdx.x; vi < nvec; vi += kSplitThreads) {
      float x[VE];
      const int cnt = load(vi, x);
#pragma unroll
      for (int i = 0; i < VE; ++i)
        if (i < cnt && in_set(x[i], vi * VE + i, lx, li)) m += elem_mass(x[i], M, c1);
    }
    return block_sum_u64(m, sh);
  }

  struct Counts {
    unsigned long long cgt, mgt, ceqb, cgt1, mgt1;
  };
  // tokens and mass above xc, tokens equal to xc before index c, tokens and mass above p1
  __device__ __noinline__ Counts counts(float xc, int64_t c, float p1) {
    const int64_t nvec = (n + VE - 1) / VE;
    unsigned long long cgt = 0, mgt = 0, ceqb = 0, cgt1 = 0, mgt1 = 0;
    for (int64_t vi = threadIdx.x; vi < nvec; vi += kSplitThreads) {
      float x[VE];
      const int cnt = load(vi, x);
#pragma unroll
      for (int i = 0; i < VE; ++i) {
        if (i >= cnt) break;
        if (x[i] > xc) {
          ++cgt;
          const unsigned long long w = elem_mass(x[i], M, c1);
          mgt += w;
          if (x[i] > p1) { ++cgt1; mgt1 += w; }
        } else if (x[i] == xc && vi * VE + i < c) {
          ++ceqb;
        }
      }
    }
    Counts o;
    o.cgt = block_sum_u64(cgt, sh);
    o.mgt = block_sum_u64(mgt, sh);
    o.ceqb = block_sum_u64(ceqb, sh);
    o.cgt1 = block_sum_u64(cgt1, sh);
    o.mgt1 = block_sum_u64(mgt1, sh);
    return o;
  }
};

template <typename T>
__global__ void __launch_bounds__(kSplitThreads) reject_sample_kernel(const Params p) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  __shared__ SplitShared sh;
  const int t = threadIdx.x;
  for (int64_t row = blockIdx.x; row < p.B; row += gridDim.x) {
    const int64_t n = p.V;
    const float temp0 = p.temperature ? p.temperature[row] : 1.f;
    const float Teff = temp0 > 0.f ? temp0 : 1.f;
    const float invT = 1.f / Teff;
    const float c1 = kLog2e * invT;
    const float topp = p.top_p ? p.top_p[row] : 1.f;
    const float minp = p.min_p ? p.min_p[row] : 0.f;
    const int32_t topk = p.top_k ? p.top_k[row] : 0;
    const bool greedy = !(temp0 > 0.f);
    int path = p.tma ? 0 : PATH_NOTMA;
    int rounds = 0;
    // ---- pass 0: maximum and non-finite check, then the mass and the count of maxima ----
    RejectRow<T> R{p, sh, row, n, 0.f, c1};
    const int64_t nvec = (n + VE - 1) / VE;
    float m = -INFINITY, mn = INFINITY, nf = 0.f;
    for (int64_t vi = t; vi < nvec; vi += kSplitThreads) {
      float x[VE];
      const int cnt = R.load(vi, x);
#pragma unroll
      for (int i = 0; i < VE; ++i)
        if (i < cnt) { m = fmaxf(m, x[i]); mn = fminf(mn, x[i]); nf = fmaf(x[i], 0.f, nf); }
    }
    const uint32_t nonfin = __syncthreads_or(nf != 0.f ? 1 : 0);
    const float M = block_max_f(m, sh);
    const float Mmin = -block_max_f(-mn, sh);
    R.M = M;
    unsigned long long s = 0;
    uint32_t cm = 0;
    int64_t first_max = 0x7FFFFFFFFFFFFFFFLL;
    if (!nonfin) {
      for (int64_t vi = t; vi < nvec; vi += kSplitThreads) {
        float x[VE];
        const int cnt = R.load(vi, x);
#pragma unroll
        for (int i = 0; i < VE; ++i) {
          if (i >= cnt) break;
          s += elem_mass(x[i], M, c1);
          if (x[i] == M) { ++cm; first_max = min(first_max, vi * VE + i); }
        }
      }
    }
    const unsigned long long Sfx = block_sum_u64(s, sh);
    const uint32_t cM = block_sum_u32(cm, sh);
    // the first maximum: the smallest index holding M
    uint32_t fm32 = first_max < n ? (uint32_t)first_max : 0xFFFFFFFFu;
    fm32 = block_min_u32(fm32, sh);
    int status = VSAMP_OK;
    if (nonfin) status = VSAMP_ERR_NONFINITE;
    else if (isnan(temp0) || isinf(temp0) || isnan(topp) || !(topp > 0.f) || isnan(minp) || minp > 1.f)
      status = VSAMP_ERR_INVALID_ARG;
    int32_t token = -1;
    float lp = __int_as_float(0x7FC00000);
    uint32_t kept_out = 0;
    const float logS = logf(u64_to_float(Sfx) * 9.094947017729282379e-13f);
    if (status == VSAMP_OK && greedy) {
      token = (int32_t)fm32;
      lp = fminf(-logS, 0.f);
      kept_out = 1;
      path |= PATH_MAXGROUP;
    } else if (status == VSAMP_OK) {
      const bool k_on = topk > 0 && (int64_t)topk < n;
      const bool p_on = topp < 1.f;
      const bool m_on = minp > 0.f;
      RowPlanner<T> P{p, sh, row, n, M, c1};
      P.Mmin = Mmin;
      // S_k: the mass the top-p target is taken on (the top-k mass when both are on)
      unsigned long long Sk = Sfx;
      if (k_on && p_on) {
        if ((unsigned long long)topk <= cM) {
          Sk = (unsigned long long)topk << kMassShift;   // k maxima, each of mass exactly 1
        } else {
          const RadixOut r = P.radix(false, (unsigned long long)topk, -1.f, true);
          const unsigned long long need = (unsigned long long)topk - r.cnt_above;
          Sk = r.mass_above + need * mass_fx(ex2_approx((Tr::value_of_rkey(r.rk) - M) * c1));
          path |= PATH_RADIX_K;
        }
      }
      const unsigned long long target_p = p_on ? ceil_mul_frac(topp, Sk) : 0ull;
      // min-p keeps x >= x*, the smallest fp32 value >= M + T ln(minp) (an unevaluated sum, as in the cut)
      float xstar = -INFINITY;
      if (m_on) {
        const float L = logf(minp);
        const float ph = Teff * L, pl_ = fmaf(Teff, L, -ph);
        const float sh_ = M + ph;
        const float bb = sh_ - M;
        const float sl = (M - (sh_ - bb)) + (ph - bb);
        const float lo = sl + pl_;
        xstar = lo > 0.f ? nextafterf(sh_, INFINITY) : sh_;
      }
      const uint64_t sd = p.seed ? p.seed[row] : 0ull;
      const uint64_t stp = p.step ? p.step[row] : 0ull;
      const uint32_t rid = p.row_id ? p.row_id[row] : (uint32_t)row;
      const PhiloxKey key{(uint32_t)sd, (uint32_t)(sd >> 32)};
      float lx = -INFINITY, high = M;
      int64_t li = 0x7FFFFFFFFFFFFFFFLL;
      unsigned long long set_mass = Sfx;
      const int cap = p.q > 0 && p.q < kRejectRounds ? p.q : kRejectRounds;   // p.q: the round cap
      for (int r = 0; r < cap && token < 0; ++r) {
        ++rounds;
        const uint32_t b = philox4x32_10(make_uint4(0xFFFFFFFFu - (uint32_t)r, rid, (uint32_t)stp, (uint32_t)(stp >> 32)),
                                         key).x;
        const unsigned long long target = __umul64hi((unsigned long long)b << 32, set_mass);   // b * mass / 2^32
        const int32_t c = R.cdf_pick(lx, li, target);
        if (c < 0) break;   // cannot happen with consistent masses: the cap path takes over
        const float xc = Tr::load_global(p.x, row * p.ld + c);
        const float p1 = 0.5f * (xc + high);
        const auto k = R.counts(xc, c, p1);
        const unsigned long long wc = elem_mass(xc, M, c1);
        const unsigned long long rank = k.cgt + k.ceqb, before = k.mgt + wc * k.ceqb;
        const bool acc = (!k_on || rank < (unsigned long long)topk) && (!p_on || before < target_p) &&
                         (!m_on || xc >= xstar);
        if (acc) {
          token = c;
          lp = fminf((xc - M) * invT - logS, 0.f);
          break;
        }
        // everything from c on in the order is outside; maybe everything at or below pivot_1 too
        lx = xc;
        li = c;
        set_mass = before;
        const bool out1 = (k_on && k.cgt1 >= (unsigned long long)topk) || (p_on && k.mgt1 >= target_p) ||
                          (m_on && p1 < xstar);
        if (out1 && p1 > xc) {
          lx = p1;
          li = -1;
          set_mass = k.mgt1;
        } else if (!out1) {
          high = p1;
        }
      }
      if (token < 0) {
        // the cap: the exact cut, then one CDF draw inside it
        path |= PATH_REJECT_CAP;
        int plan_status = VSAMP_OK;
        const Cut fin = plan_cut<T>(P, false, Teff, topk, topp, minp, Sfx, cM, path, plan_status);
        if (plan_status == VSAMP_OK) {
          float xP = Tr::value_of_rkey(fin.rk);
          int32_t It;
          if (fin.whole) It = kAllIndex;
          else It = P.nth_equal(xP, fin.need, 0);
          if (fin.whole && fin.above == 0 && fin.cnt_eq == 0) xP = -INFINITY;
          if (It >= 0) {
            const uint32_t b = philox4x32_10(make_uint4(0xFFFFFFFFu - (uint32_t)kRejectRounds, rid, (uint32_t)stp,
                                                        (uint32_t)(stp >> 32)), key).x;
            // the kept prefix's fixed-point mass, summed over the prefix itself (a top-k cut alone does not total it)
            const int64_t li_cut = It == kAllIndex ? 0x7FFFFFFFFFFFFFFFLL : (int64_t)It + 1;
            const unsigned long long mass = R.set_mass(xP, li_cut);
            const int32_t c = R.cdf_pick(xP, li_cut, __umul64hi((unsigned long long)b << 32, mass));
            if (c >= 0) {
              token = c;
              lp = fminf((Tr::load_global(p.x, row * p.ld + c) - M) * invT - logS, 0.f);
            }
          }
        }
        if (token < 0) status = VSAMP_ERR_INVALID_ARG;
      }
      kept_out = 0;   // the rejection sampler does not form the cut: the kept count is not known
    }
    if (t == 0) {
      p.token[row] = status == VSAMP_OK ? token : -1;
      if (p.logprob) p.logprob[row] = status == VSAMP_OK ? lp : __int_as_float(0x7FC00000);
      if (p.row_status) p.row_status[row] = status;
      if (p.stats) {
        p.stats[row * 4 + 0] = 2 + 2 * rounds;  // passes over the row (statistics: 2; each round: 2)
        p.stats[row * 4 + 1] = rounds;          // rejection rounds
        p.stats[row * 4 + 2] = (int32_t)kept_out;
        p.stats[row * 4 + 3] = path;
      }
    }
    __syncthreads();
  }
}

template <typename T>
vsamp_status launch_reject(Params p, int64_t B, cudaStream_t stream) {
  const int64_t rows = B < 0x7FFFFFFF ? B : 0x7FFFFFFF;
  p.q = env_int("VSAMP_REJECT_ROUNDS", kRejectRounds);   // a smaller cap (tests of the cap's fallback)
  reject_sample_kernel<T><<<(unsigned)rows, kSplitThreads, 0, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
  return VSAMP_OK;
}

}  // namespace vsamp
