// Row statistics by streaming pieces (vsamp_softmax_lse, and vsamp_logprob when it recomputes them).
//
// One thread-block cluster of C CTAs per row; the row's 4 KB pieces are split into C contiguous ranges. Every
// warp of a CTA streams its pieces through a ring of 4 KB shared-memory buffers (bulk copies issued ahead,
// bounded mbarrier waits) and writes each piece's record head straight into CTA 0's shared memory: the piece
// maximum m_p and the piece's mass relative to its own maximum in 2^-40 fixed point (the streaming sampler's
// record, by the same code, without the count of maxima and the minimum). No pass waits for the row maximum, so loads and
// arithmetic overlap across the warps of an SM. After one cluster barrier CTA 0 folds the records as the
// streaming sampler's finish does:
//   M = max_p m_p,  S = sum_p round(s_p * 2^((m_p - M) c1))  (binary64 rescale per piece, an integer sum),
// so the result depends only on the row and the piece size, not on C or on the launch.
#pragma once

#include <cooperative_groups.h>

#include <mutex>

#include "vsamp_split.cuh"

namespace vsamp {

constexpr int kStatMaxPieces = 384;   // pieces of a row this kernel takes (1.5 MB of logits)

// Shared memory of a statistics CTA of NW warps with NB piece buffers per warp.
template <int NW, int NB>
struct StatSmem {
  unsigned long long bar[NW][NB];             // per warp and buffer: the piece has landed
  uint4 gather[kStatMaxPieces];               // CTA 0: the head {m, cnt, s} of every piece's record
  float f[NW];
  uint32_t u[NW];
  unsigned long long q[NW];
  __align__(128) uint4 buf[NW][NB][kPieceBytes / 16];
};

// Launch shape of the statistics kernel for rows of V elements: pieces per row and CTAs per row (0 when a row
// has more pieces than the kernel takes).
struct StatShape {
  int np;     // pieces per row
  int C;      // CTAs per row (cluster size)
  int ppc;    // pieces per CTA (the last CTA may hold fewer)
};

// slots: CTAs resident at once on the device. A batch that fills them gets about 24 pieces per CTA (many short
// CTAs, an even spread); a smaller one gets as many CTAs per row as fit at once (one wave). At most 8 CTAs per
// row (a portable cluster), at least one piece per CTA.
inline StatShape stat_shape(int64_t V, int esize, int64_t B, int64_t slots) {
  StatShape s{0, 0, 0};
  const int64_t np = split_nchunks(V, esize);
  if (np < 1 || np > kStatMaxPieces) return s;
  int64_t C = B >= slots ? (np + 23) / 24 : slots / (B > 0 ? B : 1);
  const int forced = env_int("VSAMP_STATS_C", 0);
  if (forced > 0) C = forced;
  if (C > 8) C = 8;
  if (C < 1) C = 1;
  if (C > np) C = np;
  const int64_t ppc = (np + C - 1) / C;
  C = (np + ppc - 1) / ppc;   // no CTA without pieces
  s.np = (int)np;
  s.C = (int)C;
  s.ppc = (int)ppc;
  return s;
}

// MODE_LSE: row_max, row_logsum. MODE_LOGPROB: the log-probability of token_in[row]. Rows p.row0 + blockIdx.y.
// NW warps per CTA, NB bulk copies in flight per warp (a ring of NB buffers).
template <typename T, int MODE, int NW, int NB>
__global__ void __launch_bounds__(NW * 32, (NW >= 8 ? 3 : 6)) stats_kernel(const Params p, int np, int ppc) {
  using Tr = Traits<T>;
  using Smem = StatSmem<NW, NB>;
  extern __shared__ __align__(128) unsigned char dyn[];
  Smem& S = *reinterpret_cast<Smem*>(dyn);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int crank = blockIdx.x;
  const int64_t row = p.row0 + blockIdx.y;
  const int p0 = crank * ppc;
  const int p1 = min(np, p0 + ppc);
  cg::cluster_group cluster = cg::this_cluster();
  uint4* heads = cluster.map_shared_rank(&S.gather[0], 0);   // CTA 0's record heads (generic address)
  if (t < NW * NB) mbar_init(&S.bar[t / NB][t % NB], 1);
  fence_mbar_init();
  __syncthreads();

  const unsigned char* xr = p.x + row * p.ld * Tr::ESIZE;
  auto full_piece = [&](int pc) -> bool { return p.tma && (int64_t)(pc + 1) * kPieceElems<T> <= p.V; };
  // this warp's pieces: p0 + warp + i * NW, i < nw
  const int nw = p1 - p0 > warp ? (p1 - p0 - warp + NW - 1) / NW : 0;
  uint32_t armed = 0u, inflight = 0u, phase = 0u;   // bit b: buffer b
  bool dead = false;   // a load wait ran out: no more bulk copies from this warp
  // the bulk copy of this warp's i-th piece (a full piece of an aligned row) into buffer i % NB
  auto issue = [&](int i) {
    const int pc = p0 + warp + i * NW;
    if (dead || i >= nw || !full_piece(pc)) return;
    const int b = i % NB;
    if (lane == 0) {
      fence_proxy_async_shared();
      mbar_arrive_expect_tx(&S.bar[warp][b], (uint32_t)kPieceBytes);
      if (!p.drop_loads)
        bulk_copy_g2s(&S.buf[warp][b][0], xr + (int64_t)pc * kPieceBytes, (uint32_t)kPieceBytes, &S.bar[warp][b]);
    }
    armed |= 1u << b;
    if (!p.drop_loads) inflight |= 1u << b;
  };
#pragma unroll
  for (int i = 0; i < NB; ++i) issue(i);
  // the row's temperature is read while the first pieces land
  const float temp0 = p.temperature ? p.temperature[row] : 1.f;
  const float Teff = temp0 > 0.f ? temp0 : 1.f;   // T <= 0 (greedy) reads as T = 1
  const float invT = 1.f / Teff;
  const float c1 = kLog2e * invT;

  // ---- every warp streams its pieces ----
  for (int i = 0; i < nw; ++i) {
    const int pc = p0 + warp + i * NW;
    const int b = i % NB;
    bool timeout = false;
    const uint4* sbuf = nullptr;
    if ((armed >> b) & 1u) {
      armed &= ~(1u << b);
      if (mbar_wait_bounded(&S.bar[warp][b], (phase >> b) & 1u, p.wait_cycles)) {
        phase ^= 1u << b;
        inflight &= ~(1u << b);
        sbuf = &S.buf[warp][b][0];
      } else {
        timeout = true;
        dead = true;
      }
    }
    timeout = __any_sync(kFullMask, timeout);
    PieceRec* rec = reinterpret_cast<PieceRec*>(heads + pc);
    if (sbuf)
      piece_pass_full<T, true>(sbuf, (int64_t)pc * kPieceElems<T>, c1, timeout, false, 0u, 0u, 0u, 0u, 0u, rec,
                               nullptr);
    else
      piece_stats_partial<T, true>(xr, p.V, p.tma, (int64_t)pc * kPieceElems<T>, c1, timeout, rec);
    __syncwarp();   // every lane has finished reading buffer b
    issue(i + NB);
  }
  // a bulk copy of this warp that may still be landing (after a timed-out wait)
  for (int b = 0; b < NB; ++b)
    if ((inflight >> b) & 1u) (void)mbar_wait_bounded(&S.bar[warp][b], (phase >> b) & 1u, 4000000000LL);

  // ---- every record head is in CTA 0 once the cluster has met ----
  cluster.sync();
  if (crank != 0) return;   // nothing reads this CTA's shared memory any more

  // ---- CTA 0: M and the flags, then S rescaled to M ----
  float m = -INFINITY;
  uint32_t flags = 0;   // 1: a non-finite value, 2: a load timed out
  for (int i = t; i < np; i += NW * 32) {
    const uint4 h = S.gather[i];
    const float mp = __uint_as_float(h.x);
    if (mp != mp) flags |= h.y == kTimeoutCnt ? 3u : 1u;
    else m = fmaxf(m, mp);
  }
  m = warp_max_f(m);
  flags = __reduce_or_sync(kFullMask, flags);
  if (lane == 0) { S.f[warp] = m; S.u[warp] = flags; }
  __syncthreads();
  float M = S.f[0];
  flags = S.u[0];
#pragma unroll
  for (int w = 1; w < NW; ++w) { M = fmaxf(M, S.f[w]); flags |= S.u[w]; }
  unsigned long long Sp = 0;
  if (!flags) {
    for (int i = t; i < np; i += NW * 32) {
      const uint4 h = S.gather[i];
      const float mp = __uint_as_float(h.x);
      const unsigned long long sp = ((unsigned long long)h.w << 32) | h.z;
      if (mp == M) {
        Sp += sp;
      } else {
        // 2^((m_p - M) * c1) is below 1: the piece's fixed-point mass rescaled in binary64
        const double f = exp2((double)((mp - M) * c1));
        Sp += (unsigned long long)__double2ull_rn((double)sp * f);
      }
    }
  }
  Sp = warp_sum_u64(Sp);
  if (lane == 0) S.q[warp] = Sp;
  __syncthreads();
  if (t != 0) return;
  unsigned long long Sfx = 0;
#pragma unroll
  for (int w = 0; w < NW; ++w) Sfx += S.q[w];

  // ---- status and outputs (thread 0) ----
  int status = VSAMP_OK;
  if (flags & 2u) status = VSAMP_ERR_TIMEOUT;
  else if (flags) status = VSAMP_ERR_NONFINITE;
  else if (isnan(temp0) || isinf(temp0)) status = VSAMP_ERR_INVALID_ARG;
  int32_t tok = 0;
  if ((MODE & MODE_LOGPROB) && status == VSAMP_OK) {
    tok = p.token_in[row];
    if (tok < 0 || (int64_t)tok >= p.V) status = VSAMP_ERR_INVALID_ARG;
  }
  const float logS = logf(u64_to_float(Sfx) * 9.094947017729282379e-13f);   // 2^-40
  if (MODE & MODE_LSE) {
    if (p.row_max) p.row_max[row] = status == VSAMP_OK ? M : __int_as_float(0x7FC00000);
    if (p.row_logsum) p.row_logsum[row] = status == VSAMP_OK ? logS : __int_as_float(0x7FC00000);
  }
  if (MODE & MODE_LOGPROB) {
    float lp = __int_as_float(0x7FC00000);
    if (status == VSAMP_OK) lp = fminf((Tr::load_global(xr, tok) - M) * invT - logS, 0.f);
    if (p.logprob) p.logprob[row] = lp;
  }
  if (p.row_status) p.row_status[row] = status;
}

// Host: one launch per 65,535 rows, clusters of C CTAs over grid (C, rows), NW warps and NB buffers per warp.
template <typename T, int MODE, int NW, int NB>
static vsamp_status launch_stats_cfg(Params p, int64_t B, int esize, const DeviceInfo& d, int dev,
                                     cudaStream_t stream) {
  static int ready[64] = {0};
  static std::mutex mu;
  auto kern = stats_kernel<T, MODE, NW, NB>;
  const int smem = (int)sizeof(StatSmem<NW, NB>);
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!ready[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ready[dev], kern, NW * 32, smem) != cudaSuccess) {
        cudaGetLastError();
        ready[dev] = 0;
        return VSAMP_ERR_UNSUPPORTED;
      }
    }
    per_sm = ready[dev];
  }
  if (per_sm < 1) return VSAMP_ERR_UNSUPPORTED;
  const StatShape sh = stat_shape(p.V, esize, B, (int64_t)per_sm * d.sm_count);
  if (sh.np == 0) return VSAMP_ERR_UNSUPPORTED;
  const long long wc = env_ll("VSAMP_WAIT_CYCLES", 0);
  p.wait_cycles = wc > 0 ? wc : 4000000000LL;   // ~2 s at the maximum SM clock
  p.drop_loads = env_int("VSAMP_TEST_DROP_LOADS", 0) != 0 ? 1 : 0;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(NW * 32, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)sh.C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  for (int64_t r0 = 0; r0 < B; r0 += 65535) {
    const int64_t nb = B - r0 < 65535 ? B - r0 : 65535;
    p.row0 = r0;
    cfg.gridDim = dim3((unsigned)sh.C, (unsigned)nb, 1);
    if (cudaLaunchKernelEx(&cfg, kern, p, sh.np, sh.ppc) != cudaSuccess) {
      cudaGetLastError();
      return VSAMP_ERR_CUDA;
    }
  }
  return VSAMP_OK;
}

// VSAMP_ERR_UNSUPPORTED when the rows are longer than the kernel takes (the caller then uses the cluster row
// kernel).
template <typename T, int MODE>
vsamp_status launch_stats(Params p, int64_t B, int esize, cudaStream_t stream) {
  if (split_nchunks(p.V, esize) > kStatMaxPieces) return VSAMP_ERR_UNSUPPORTED;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return VSAMP_ERR_CUDA; }
  if (dev < 0 || dev >= 64) return VSAMP_ERR_UNSUPPORTED;
  DeviceInfo d;
  const vsamp_status ds = device_info(dev, d);
  if (ds != VSAMP_OK) return ds;
  switch (env_int("VSAMP_STATS_CFG", 0)) {
    // other (warps, buffers) shapes, for measurements
    case 1: return launch_stats_cfg<T, MODE, 8, 2>(p, B, esize, d, dev, stream);
    case 2: return launch_stats_cfg<T, MODE, 8, 1>(p, B, esize, d, dev, stream);
    default: return launch_stats_cfg<T, MODE, 4, 2>(p, B, esize, d, dev, stream);
  }
}

}  // namespace vsamp
