// Vocabulary-sharded sampling (vsamp_shard_partial, vsamp_shard_merge): each shard of a row's vocabulary writes
// rank-local summaries -- the 4 KB piece records of the streaming sampler and the shard's own certified Gumbel-max
// winner -- which are exchanged by an all-gather in rank order (no reduction in transit) and merged by one owned,
// fixed fold ("[WS2][Logprob] Deterministic SM90 linear_logp ...", Tensor parallelism: rank order + owned merge).
//   partial  the piece pass over the shard (Philox counters from the tokens' global indices), then one CTA per row
//            combines the shard's pieces relative to the shard maximum m_r, and draws the shard's winner over all
//            of its tokens: the vectors whose draw code passes the prune bound of the shard's own mass, scored
//            exactly, certified against that bound (the shard's tokens are scanned when it does not hold).
//   merge    one CTA per row: the global maximum (order-free), the piece masses rescaled to it and summed as
//            integers (so the result does not depend on the order, the shard count, or -- for shard boundaries on
//            piece boundaries -- on the sharding at all), log S, then the winner: max and arg-max decompose over
//            shards, so the arg-max of the shards' winners under the global scores (x - M) / T + g is the
//            unsharded draw. The selected token's log-probability comes from its single owner.
// The draw is over the full temperature-scaled distribution: filters (top-k, top-p, min-p) need the cut, which
// depends on the whole row, and are not part of the sharded entry points.
#pragma once

#include "vsamp_split.cuh"

namespace vsamp {

struct ShardWin {          // vsamp_shard_win: 16 bytes per (row, shard)
  int32_t idx;             // the shard's winner, global index (-1 on a row error)
  float x;                 // its logit
  float xt;                // the target token's logit when the shard owns it
  int32_t flags;           // bit 0: owns the target; bits 8..15: the shard's row status
};
static_assert(sizeof(ShardWin) == 16, "ShardWin layout");

// One CTA per row: the shard's winner from its piece records (rows blockIdx.x, blockIdx.x + gridDim.x, ...).
template <typename T>
__global__ void __launch_bounds__(kStreamThreads) shard_finish_kernel(const Params p, const StreamWs ws, int np,
                                                                      const int32_t* target, ShardWin* win) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  __shared__ FinishSmem S;
  SplitShared& sh = S.sh;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int64_t n = p.V;   // the shard's length
  for (int64_t row = blockIdx.x; row < p.B; row += gridDim.x) {
    PieceRec* recs = ws.recs + row * ws.rec_ld;
    // the record slots past the shard's pieces hold empty records (maximum -inf, no mass)
    for (int64_t k = np + t; k < ws.rec_ld; k += kStreamThreads) {
      uint4* o = reinterpret_cast<uint4*>(recs + k);
      o[0] = make_uint4(__float_as_uint(-INFINITY), 0u, 0u, 0u);
      o[1] = make_uint4(__float_as_uint(INFINITY), 0u, 0u, 0u);
    }
    const float temp0 = p.temperature ? p.temperature[row] : 1.f;
    const float Teff = temp0 > 0.f ? temp0 : 1.f;
    const float invT = 1.f / Teff;
    const float c1 = kLog2e * invT;
    const int64_t nwords = (int64_t)np * 32;
    const bool greedy = !(temp0 > 0.f);
    const bool staged = !greedy && nwords <= (int64_t)kCodeSmem;
    if (staged) {
      const uint32_t* src = ws.codes + row * nwords;
#pragma unroll 4
      for (int w = t; w < (int)nwords; w += kStreamThreads) S.codes[w] = __ldcg(src + w);
    }
    // ---- the shard's maximum, flags, mass relative to its maximum ----
    float m = -INFINITY;
    uint32_t flags = 0;
    for (int k = t; k < np; k += kStreamThreads) {
      const PieceRec r = load_rec(recs + k);
      if (r.m != r.m) flags |= r.cnt == kTimeoutCnt ? 3u : 1u;
      else m = fmaxf(m, r.m);
    }
    m = warp_max_f(m);
    flags = __reduce_or_sync(kFullMask, flags);
    __syncthreads();
    if (lane == 0) { sh.f[warp] = m; sh.u[warp][0] = flags; }
    __syncthreads();
    float Mr = sh.f[0];
    flags = sh.u[0][0];
#pragma unroll
    for (int w = 1; w < kItemPieces; ++w) { Mr = fmaxf(Mr, sh.f[w]); flags |= sh.u[w][0]; }
    unsigned long long Sp = 0;
    int kfirst = 0x7FFFFFFF;   // the first piece holding the shard maximum
    for (int k = t; k < np; k += kStreamThreads) {
      const PieceRec r = load_rec(recs + k);
      if (r.m == Mr) {
        Sp += r.s;
        kfirst = min(kfirst, k);
      } else if (!flags) {
        Sp += (unsigned long long)__double2ull_rn((double)r.s * exp2((double)((r.m - Mr) * c1)));
      }
    }
    Sp = warp_sum_u64(Sp);
    kfirst = (int)__reduce_min_sync(kFullMask, (uint32_t)kfirst);
    if (lane == 0) { sh.q[warp][0] = Sp; sh.u[warp][1] = (uint32_t)kfirst; }
    __syncthreads();
    unsigned long long Sfx = 0;
    uint32_t kf = 0xFFFFFFFFu;
#pragma unroll
    for (int w = 0; w < kItemPieces; ++w) { Sfx += sh.q[w][0]; kf = min(kf, sh.u[w][1]); }
    int status = VSAMP_OK;
    if (flags & 2u) status = VSAMP_ERR_TIMEOUT;
    else if (flags) status = VSAMP_ERR_NONFINITE;
    else if (isnan(temp0) || isinf(temp0)) status = VSAMP_ERR_INVALID_ARG;
    int32_t idx_local = -1;
    if (status == VSAMP_OK && greedy) {
      // the shard's first maximum
      if (warp == 0) {
        const PieceView<T> pv{p.x + row * p.ld * Tr::ESIZE, n, p.tma, (int64_t)kf * kPieceElems<T>};
        const int32_t f = piece_nth_equal_staged<T>(pv, Mr, 1u, S.piece);
        if (lane == 0) S.it = f;
      }
      __syncthreads();
      idx_local = S.it;
    } else if (status == VSAMP_OK) {
      const float sr = fmaxf(u64_to_float(Sfx) * 9.094947017729282379e-13f, 1.f);
      DrawRow d;
      d.M = Mr;
      d.invT = invT;
      d.c1 = c1;
      d.xP = -INFINITY;
      d.It = kAllIndex;
      d.kappa = 20.085536923187668f / sr;
      d.all_cand = d.kappa >= 0.99f;
      d.bk = d.all_cand ? 0xFFFFFFFFu : __float2uint_ru(d.kappa * 1.00001f * 4294967296.0f);
      const uint64_t sd = p.seed ? p.seed[row] : 0ull;
      const uint64_t stp = p.step ? p.step[row] : 0ull;
      d.rid = p.row_id ? p.row_id[row] : (uint32_t)row;
      d.st_lo = (uint32_t)stp;
      d.st_hi = (uint32_t)(stp >> 32);
      d.key = PhiloxKey{(uint32_t)sd, (uint32_t)(sd >> 32)};
      const float B0 = -logf(d.kappa);
      float bscore = -INFINITY, bs = 0.f;
      int32_t bidx = 0x7FFFFFFF;
      bool done = false;
      if (staged && !d.all_cand) {
        if (t == 0) S.nflag = 0u;
        __syncthreads();
        const uint32_t cbk = draw_code(d.bk);
        const uint32_t addk = (16u - cbk) * 0x01010101u;
        const int64_t nvec = (n + VE - 1) / VE;
#pragma unroll 1
        for (int w = t; w < (int)nwords; w += kStreamThreads) {
          const uint32_t word = S.codes[w];
          const uint32_t ge = (((word & 0x0F0F0F0Fu) + addk) & 0x10101010u) |
                              ((((word >> 4) & 0x0F0F0F0Fu) + addk) & 0x10101010u);
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
        const uint32_t nflag = S.nflag;
        if (nflag <= (uint32_t)kFlagMax) {
          const unsigned char* xr = p.x + row * p.ld * Tr::ESIZE;
          for (uint32_t i = t; i < nflag; i += kStreamThreads) {
            const int64_t e0 = (int64_t)S.flist[i] * VE;
            uint4 v;
            const int cnt = load_vec<T, false>(p, xr, e0, v);
            score_vector<T>(v, cnt, p.v0 + e0, d, bscore, bidx, bs);
          }
          done = true;
        }
      }
      if (!done) score_row<T>(p, row, d, bscore, bidx, bs);
      ArgMax g = block_argmax(ArgMax{bscore, bidx, bs}, S);
      if (!(d.all_cand || (g.idx != 0x7FFFFFFF && g.score > B0 + 1e-4f * fmaxf(1.f, fabsf(B0))))) {
        DrawRow all = d;   // the bound did not certify the shard's winner: all of its tokens, exactly
        all.all_cand = true;
        bscore = -INFINITY;
        bs = 0.f;
        bidx = 0x7FFFFFFF;
        score_row<T>(p, row, all, bscore, bidx, bs);
        g = block_argmax(ArgMax{bscore, bidx, bs}, S);
      }
      idx_local = g.idx != 0x7FFFFFFF ? (int32_t)(g.idx - p.v0) : -1;
    }
    if (t == 0) {
      ShardWin o;
      o.idx = -1;
      o.x = __int_as_float(0x7FC00000);
      o.xt = __int_as_float(0x7FC00000);
      o.flags = 0;
      if (status == VSAMP_OK && (idx_local < 0 || (int64_t)idx_local >= n)) status = VSAMP_ERR_INVALID_ARG;
      if (status == VSAMP_OK) {
        o.idx = (int32_t)(p.v0 + idx_local);
        o.x = Tr::load_global(p.x, row * p.ld + idx_local);
      }
      if (target) {
        const int64_t tl = (int64_t)target[row] - p.v0;
        if (tl >= 0 && tl < n) {
          o.flags |= 1;
          o.xt = Tr::load_global(p.x, row * p.ld + tl);
        }
      }
      o.flags |= status << 8;
      win[row] = o;
    }
    __syncthreads();
  }
}

// The owned merge: one CTA per row over the rank-ordered records [R, B, NP] and winners [R, B] (a template only so
// that the header can be included by several translation units).
template <int kUnused>
__global__ void __launch_bounds__(kStreamThreads) shard_merge_kernel(
    const PieceRec* recs, const ShardWin* wins, int R, int64_t B, int64_t NP, int64_t V, const float* temperature,
    const uint64_t* seed, const uint64_t* step, const uint32_t* row_id, float* row_max, float* row_logsum,
    int32_t* token, float* logprob, float* target_logprob, int32_t* row_status) {
  __shared__ SplitShared sh;
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  for (int64_t row = blockIdx.x; row < B; row += gridDim.x) {
    const float temp0 = temperature ? temperature[row] : 1.f;
    const float Teff = temp0 > 0.f ? temp0 : 1.f;
    const float invT = 1.f / Teff;
    const float c1 = kLog2e * invT;
    const int64_t nrec = (int64_t)R * NP;
    auto rec_of = [&](int64_t i) -> const PieceRec* { return recs + ((i / NP) * B + row) * NP + i % NP; };
    // ---- the global maximum (order-free), then the piece masses rescaled to it, summed as integers ----
    float m = -INFINITY;
    uint32_t flags = 0;
    for (int64_t i = t; i < nrec; i += kStreamThreads) {
      const PieceRec r = load_rec(rec_of(i));
      if (r.m != r.m) flags |= r.cnt == kTimeoutCnt ? 3u : 1u;
      else m = fmaxf(m, r.m);
    }
    m = warp_max_f(m);
    flags = __reduce_or_sync(kFullMask, flags);
    __syncthreads();
    if (lane == 0) { sh.f[warp] = m; sh.u[warp][0] = flags; }
    __syncthreads();
    float M = sh.f[0];
    flags = sh.u[0][0];
#pragma unroll
    for (int w = 1; w < kItemPieces; ++w) { M = fmaxf(M, sh.f[w]); flags |= sh.u[w][0]; }
    unsigned long long Sp = 0;
    for (int64_t i = t; i < nrec; i += kStreamThreads) {
      const PieceRec r = load_rec(rec_of(i));
      if (r.m == M) Sp += r.s;
      else if (!flags) Sp += (unsigned long long)__double2ull_rn((double)r.s * exp2((double)((r.m - M) * c1)));
    }
    Sp = warp_sum_u64(Sp);
    if (lane == 0) sh.q[warp][0] = Sp;
    __syncthreads();
    if (warp == 0) {
      unsigned long long Sfx = 0;
#pragma unroll
      for (int w = 0; w < kItemPieces; ++w) Sfx += sh.q[w][0];
      // ---- the shards' winners under the global scores: lane r holds shard r's ----
      int status = flags & 2u ? VSAMP_ERR_TIMEOUT : (flags ? VSAMP_ERR_NONFINITE : VSAMP_OK);
      if (status == VSAMP_OK && (isnan(temp0) || isinf(temp0))) status = VSAMP_ERR_INVALID_ARG;
      const bool greedy = !(temp0 > 0.f);
      const float logS = logf(u64_to_float(Sfx) * 9.094947017729282379e-13f);
      const uint64_t sd = seed ? seed[row] : 0ull;
      const uint64_t stp = step ? step[row] : 0ull;
      const uint32_t rid = row_id ? row_id[row] : (uint32_t)row;
      float best = -INFINITY, bs = 0.f, xt = __int_as_float(0x7FC00000);
      int32_t bidx = 0x7FFFFFFF;
      int shard_status = VSAMP_OK;
      bool owned = false;
      for (int r0 = 0; r0 < R; r0 += 32) {
        const int r = r0 + lane;
        if (r < R) {
          const ShardWin w = wins[(int64_t)r * B + row];
          const int st = (w.flags >> 8) & 0xFF;
          if (st != VSAMP_OK && shard_status == VSAMP_OK) shard_status = st;
          if (w.flags & 1) { owned = true; xt = w.xt; }
          if (st == VSAMP_OK && w.idx >= 0) {
            float score;
            const float sv = (w.x - M) * invT;
            if (greedy) {
              score = w.x == M ? 0.f : -INFINITY;   // the first maximum: the lowest index among the maxima
            } else {
              const uint4 w4 = philox4x32_10(make_uint4((uint32_t)w.idx >> 2, rid, (uint32_t)stp, (uint32_t)(stp >> 32)),
                                             PhiloxKey{(uint32_t)sd, (uint32_t)(sd >> 32)});
              score = gumbel_score(sv, philox_word(w4, w.idx & 3));
            }
            if (argmax_better(score, w.idx, best, bidx)) { best = score; bidx = w.idx; bs = sv; }
          }
        }
      }
      const ArgMax g = warp_argmax(ArgMax{best, bidx, bs});
      // the first error in rank order (every shard sees the same temperature; any non-finite value is an error)
      const uint32_t bad = __ballot_sync(kFullMask, shard_status != VSAMP_OK);
      const int first_err = bad ? __shfl_sync(kFullMask, shard_status, __ffs(bad) - 1) : VSAMP_OK;
      const uint32_t own = __ballot_sync(kFullMask, owned);
      const float xt_own = own ? __shfl_sync(kFullMask, xt, __ffs(own) - 1) : __int_as_float(0x7FC00000);
      if (status == VSAMP_OK) status = first_err;
      if (status == VSAMP_OK && !(g.idx >= 0 && (int64_t)g.idx < V)) status = VSAMP_ERR_INVALID_ARG;
      if (status == VSAMP_OK && target_logprob && !own) status = VSAMP_ERR_INVALID_ARG;   // no shard owns the target
      if (lane == 0) {
        const float nan = __int_as_float(0x7FC00000);
        const bool ok = status == VSAMP_OK;
        if (row_max) row_max[row] = ok ? M : nan;
        if (row_logsum) row_logsum[row] = ok ? logS : nan;
        if (token) token[row] = ok ? g.idx : -1;
        if (logprob) logprob[row] = ok ? fminf(g.s - logS, 0.f) : nan;
        if (target_logprob) target_logprob[row] = ok ? fminf((xt_own - M) * invT - logS, 0.f) : nan;
        if (row_status) row_status[row] = status;
      }
    }
    __syncthreads();
  }
}

}  // namespace vsamp
