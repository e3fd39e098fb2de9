// The streaming sampler without a workspace (vsamp_sample for rows of up to kFinishPieces pieces).
//
// One thread-block cluster of C CTAs per row; the row's 4 KB pieces are split into C contiguous ranges. Every
// warp streams its pieces through bulk-copy buffers and forms each piece's record and, for a row drawn over a
// possibly large kept set (T > 0, no top-k), its draw codes (the smallest Philox word of each 16-byte vector,
// data independent), exactly as the streaming sampler's piece pass does; both go straight into CTA 0's
// shared memory. After one cluster barrier the other CTAs leave and CTA 0 runs the streaming sampler's row
// finish on them: the statistics, the plan of the cut (re-reading the row from L2 only where the cut leaves
// the maximum's tie group), the boundary, and the exact scores of the code-flagged vectors. Other clusters
// keep streaming on the same SMs while a CTA 0 finishes, so the finish's latency overlaps their loads.
#pragma once

#include <cooperative_groups.h>

#include <mutex>

#include "vsamp_split.cuh"

namespace vsamp {

constexpr int kFinishPieces = kCodeSmem / 32;   // pieces of a row whose codes CTA 0 holds: 150

template <int NB>
struct SampleStreamSmem {
  unsigned long long bar[kItemPieces][NB];      // per warp and buffer: the piece has landed
  PieceRec recs[kFinishPieces];                 // CTA 0: every piece's record
  FinishSmem fin;                               // CTA 0: the row finish (its codes array holds the row's codes)
  __align__(128) uint4 buf[kItemPieces][NB][kPieceBytes / 16];
};

template <typename T, int NB>
__global__ void __launch_bounds__(kStreamThreads, 3) sample_stream_kernel(const Params p, int np, int ppc) {
  using Tr = Traits<T>;
  using Smem = SampleStreamSmem<NB>;
  extern __shared__ __align__(128) unsigned char dyn[];
  Smem& S = *reinterpret_cast<Smem*>(dyn);
  const int t = threadIdx.x, lane = t & 31, warp = t >> 5;
  const int crank = blockIdx.x;
  const int64_t row = p.row0 + blockIdx.y;
  const int p0 = crank * ppc;
  const int p1 = min(np, p0 + ppc);
  cg::cluster_group cluster = cg::this_cluster();
  Smem* s0 = cluster.map_shared_rank(&S, 0);   // CTA 0's shared memory (generic address)
  PieceRec* recs0 = &s0->recs[0];
  uint32_t* codes0 = &s0->fin.codes[0];
  if (t < kItemPieces * NB) mbar_init(&S.bar[t / NB][t % NB], 1);
  fence_mbar_init();
  __syncthreads();

  const unsigned char* xr = p.x + row * p.ld * Tr::ESIZE;
  auto full_piece = [&](int pc) -> bool { return p.tma && (int64_t)(pc + 1) * kPieceElems<T> <= p.V; };
  const int nw = p1 - p0 > warp ? (p1 - p0 - warp + kItemPieces - 1) / kItemPieces : 0;
  uint32_t armed = 0u, inflight = 0u, phase = 0u;   // bit b: buffer b
  bool dead = false;                                // a load wait ran out: no more bulk copies from this warp
  auto issue = [&](int i) {
    const int pc = p0 + warp + i * kItemPieces;
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
  // the row's parameters are read while the first pieces land
  const float temp0 = p.temperature ? p.temperature[row] : 1.f;
  const float c1 = kLog2e * (1.f / (temp0 > 0.f ? temp0 : 1.f));
  const bool coded = row_coded(p, row) && np <= kFinishPieces;
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

  // ---- every warp streams its pieces: the record and the codes into CTA 0 ----
  for (int i = 0; i < nw; ++i) {
    const int pc = p0 + warp + i * kItemPieces;
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
    const int64_t e_begin = (int64_t)pc * kPieceElems<T>;
    if (sbuf) {
      piece_pass_full<T>(sbuf, e_begin, c1, timeout, coded, k0, k1, rid, st_lo, st_hi, recs0 + pc, codes0 + pc * 32);
    } else {
      piece_stats_partial<T>(xr, p.V, p.tma, e_begin, c1, timeout, recs0 + pc);
      if (coded && !timeout) piece_codes<T>(e_begin, k0, k1, rid, st_lo, st_hi, codes0 + pc * 32);
    }
    __syncwarp();   // every lane has finished reading buffer b
    issue(i + NB);
  }
  // a bulk copy of this warp that may still be landing (after a timed-out wait)
  for (int b = 0; b < NB; ++b)
    if ((inflight >> b) & 1u) (void)mbar_wait_bounded(&S.bar[warp][b], (phase >> b) & 1u, 4000000000LL);

  // ---- every record and code is in CTA 0 once the cluster has met; CTA 0 finishes the row ----
  cluster.sync();
  if (crank != 0) return;   // nothing reads this CTA's shared memory any more
  finish_row<T, true>(p, StreamWs{&S.recs[0], 0, &S.fin.codes[0]}, row, np, S.fin);
}

// Host: one launch per 65,535 rows, clusters of C CTAs over grid (C, rows). VSAMP_ERR_UNSUPPORTED when a row has
// more pieces than CTA 0 holds (the caller then uses the cluster sampling kernel).
template <typename T, int NB>
static vsamp_status launch_sample_stream_cfg(Params p, int64_t B, int esize, const DeviceInfo& d, int dev,
                                             cudaStream_t stream) {
  static int ready[64] = {0};
  static std::mutex mu;
  auto kern = sample_stream_kernel<T, NB>;
  const int smem = (int)sizeof(SampleStreamSmem<NB>);
  int per_sm = 0;
  {
    std::lock_guard<std::mutex> lk(mu);
    if (!ready[dev]) {
      if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess ||
          cudaOccupancyMaxActiveBlocksPerMultiprocessor(&ready[dev], kern, kStreamThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        ready[dev] = 0;
        return VSAMP_ERR_UNSUPPORTED;
      }
    }
    per_sm = ready[dev];
  }
  if (per_sm < 1) return VSAMP_ERR_UNSUPPORTED;
  const int64_t np = split_nchunks(p.V, esize);
  if (np < 1 || np > kFinishPieces) return VSAMP_ERR_UNSUPPORTED;
  // a batch that fills the resident slots gets about 24 pieces per CTA; a smaller one as many CTAs per row as
  // fit at once; at most 8 (a portable cluster), at least one piece per CTA
  const int64_t slots = (int64_t)per_sm * d.sm_count;
  int64_t C = B >= slots ? (np + 23) / 24 : slots / (B > 0 ? B : 1);
  const int forced = env_int("VSAMP_SSTREAM_C", 0);
  if (forced > 0) C = forced;
  if (C > 8) C = 8;
  if (C < 1) C = 1;
  if (C > np) C = np;
  const int64_t ppc = (np + C - 1) / C;
  C = (np + ppc - 1) / ppc;
  const long long wc = env_ll("VSAMP_WAIT_CYCLES", 0);
  p.wait_cycles = wc > 0 ? wc : 4000000000LL;   // ~2 s at the maximum SM clock
  p.drop_loads = env_int("VSAMP_TEST_DROP_LOADS", 0) != 0 ? 1 : 0;
  p.v0 = 0;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(kStreamThreads, 1, 1);
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  for (int64_t r0 = 0; r0 < B; r0 += 65535) {
    const int64_t nb = B - r0 < 65535 ? B - r0 : 65535;
    p.row0 = r0;
    cfg.gridDim = dim3((unsigned)C, (unsigned)nb, 1);
    if (cudaLaunchKernelEx(&cfg, kern, p, (int)np, (int)ppc) != cudaSuccess) {
      cudaGetLastError();
      return VSAMP_ERR_CUDA;
    }
  }
  return VSAMP_OK;
}

template <typename T>
vsamp_status launch_sample_stream(Params p, int64_t B, int esize, cudaStream_t stream) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) { cudaGetLastError(); return VSAMP_ERR_CUDA; }
  if (dev < 0 || dev >= 64) return VSAMP_ERR_UNSUPPORTED;
  DeviceInfo d;
  const vsamp_status ds = device_info(dev, d);
  if (ds != VSAMP_OK) return ds;
  if (env_int("VSAMP_SSTREAM_NB", 1) == 2) return launch_sample_stream_cfg<T, 2>(p, B, esize, d, dev, stream);
  return launch_sample_stream_cfg<T, 1>(p, B, esize, d, dev, stream);
}

}  // namespace vsamp
