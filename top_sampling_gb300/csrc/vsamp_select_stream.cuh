// The uncached top-k select (vsamp_topk_select for rows longer than a thread-block cluster holds on chip):
// one CTA per row reads the row from global memory at every pass ("[Kernel] Make persistent_topk deterministic",
// the wide-row fallback: an uncached path for rows that do not fit). The result is that of the on-chip select:
//   pass 0   NaN check inside the row's length (a data error, reported before a k > k_max error);
//   radix    the count search over the order-preserving key, 8 bits per round (4 rounds fp32, 2 bf16), each
//            round a 256-bin histogram of the keys matching the prefix found so far, re-read from L2 / HBM;
//   emission the keys above the pivot and the lowest-index `need` keys equal to it, written in ascending index
//            order: tiles of 256 vectors, one block scan of the equal counts (which of them are taken) and one of
//            the taken counts (where they go) per tile.
#pragma once

#include "vsamp_split.cuh"

namespace vsamp {

template <typename T>
__global__ void __launch_bounds__(kSplitThreads) select_stream_kernel(const Params p) {
  using Tr = Traits<T>;
  constexpr int VE = Tr::VE;
  __shared__ SplitShared sh;
  const int t = threadIdx.x;
  for (int64_t row = blockIdx.x; row < p.B; row += gridDim.x) {
    int32_t* orow = p.out_idx + row * (int64_t)p.k_max;
    int64_t n = p.lengths ? (int64_t)p.lengths[row] : p.V;
    const bool bad_len = !(n > 0 && n <= p.V);
    if (bad_len) n = 0;
    const int32_t k = p.k_sel ? p.k_sel[row] : p.k_max;
    const unsigned char* xr = p.x + row * p.ld * Tr::ESIZE;
    const int64_t nvec = (n + VE - 1) / VE;
    // ---- NaN inside the length; the range of the values (the radix search's first round) ----
    uint32_t nan = 0;
    float mx = -INFINITY, mn = INFINITY;
    for (int64_t vi = t; vi < nvec; vi += kSplitThreads) {
      uint4 v;
      int cnt = load_vec<T, false>(p, xr, vi * VE, v);
      if (n - vi * VE < cnt) cnt = (int)(n - vi * VE);   // the row's own length, not the batch's
      float x[VE];
      Tr::values(v, x);
#pragma unroll
      for (int i = 0; i < VE; ++i) {
        if (i < cnt) {
          nan |= x[i] != x[i] ? 1u : 0u;
          mx = fmaxf(mx, x[i]);
          mn = fminf(mn, x[i]);
        }
      }
    }
    nan = __syncthreads_or(nan);
    const float Mrow = block_max_f(mx, sh);
    const float Mmin = -block_max_f(-mn, sh);
    int status = VSAMP_OK;
    if (bad_len) status = VSAMP_ERR_INVALID_ARG;
    else if (nan) status = VSAMP_ERR_NONFINITE;
    else if (k > p.k_max) status = VSAMP_ERR_INVALID_ARG;
    int64_t total = 0;
    if (status == VSAMP_OK && k > 0) {
      float xP = -INFINITY;
      unsigned long long need = 0;
      bool all = (int64_t)k >= n;
      if (!all) {
        RowPlanner<T> P{p, sh, row, n, Mrow, 0.f};
        P.Mmin = Mmin;
        const RadixOut r = P.radix(false, (unsigned long long)k, -1.f, false);
        if (!r.ok) {
          status = VSAMP_ERR_INVALID_ARG;   // cannot happen with consistent counts
        } else {
          xP = Tr::value_of_rkey(r.rk);
          need = (unsigned long long)k - r.cnt_above;
        }
      }
      if (status == VSAMP_OK) {
        // ---- emission in ascending index order ----
        unsigned long long eq_base = 0;
        for (int64_t v0 = 0; v0 < nvec; v0 += kSplitThreads) {
          const int64_t vi = v0 + t;
          float x[VE];
          int cnt = 0;
          if (vi < nvec) {
            uint4 v;
            cnt = load_vec<T, false>(p, xr, vi * VE, v);
            if (n - vi * VE < cnt) cnt = (int)(n - vi * VE);
            Tr::values(v, x);
          }
          uint32_t c_eq = 0;
#pragma unroll
          for (int i = 0; i < VE; ++i) c_eq += (i < cnt && !all && x[i] == xP) ? 1u : 0u;
          uint32_t eq_tot;
          const uint32_t eq_pre = block_scan_u32(c_eq, eq_tot, sh);
          // this thread's equal keys start at rank eq_base + eq_pre among the row's keys equal to the pivot
          uint32_t sel = 0;
          {
            unsigned long long eq_rank = eq_base + eq_pre;
#pragma unroll
            for (int i = 0; i < VE; ++i) {
              if (i >= cnt) break;
              if (all || x[i] > xP) ++sel;
              else if (x[i] == xP) { if (eq_rank < need) ++sel; ++eq_rank; }
            }
          }
          uint32_t sel_tot;
          const uint32_t sel_pre = block_scan_u32(sel, sel_tot, sh);
          if (sel) {
            int64_t pos = total + sel_pre;
            unsigned long long eq_rank = eq_base + eq_pre;
#pragma unroll
            for (int i = 0; i < VE; ++i) {
              if (i >= cnt) break;
              bool take = all || x[i] > xP;
              if (!take && x[i] == xP) { take = eq_rank < need; ++eq_rank; }
              if (take) {
                if (pos < p.k_max) orow[pos] = (int32_t)(vi * VE + i);
                ++pos;
              }
            }
          }
          total += sel_tot;
          eq_base += eq_tot;
        }
      }
    }
    if (status != VSAMP_OK) total = 0;
    for (int64_t j = total + t; j < p.k_max; j += kSplitThreads) orow[j] = -1;
    if (t == 0 && p.row_status) p.row_status[row] = status;
    __syncthreads();
  }
}

template <typename T>
vsamp_status launch_select_stream(Params p, int64_t B, cudaStream_t stream) {
  const int64_t rows = B < 0x7FFFFFFF ? B : 0x7FFFFFFF;
  select_stream_kernel<T><<<(unsigned)rows, kSplitThreads, 0, stream>>>(p);
  if (cudaGetLastError() != cudaSuccess) return VSAMP_ERR_CUDA;
  return VSAMP_OK;
}

}  // namespace vsamp
