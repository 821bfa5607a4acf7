// Range-table fill on the GPU.
//
// Restates vLLM PR #50294 review, "Key source snippets",
// fill_mm_prefix_query_ranges, as a data-parallel integer kernel: one thread
// per packed query row.  The thread finds its request by binary search over
// query_start_loc, forms the row's absolute position ctx + local, and scans
// the request's ranges in list order, keeping the last valid (start < end)
// closed range that holds the position -- exactly the row the page's span
// writes would leave behind, since later spans overwrite earlier ones and a
// span covers precisely the rows whose position lies in [start, end] within
// the scheduled chunk.  Every row [0, num_tokens) is written (unlike the page,
// which leaves the buffer untouched when nothing is covered), and
// rows_written receives the page's return value.  Rows at or past
// query_start_loc[num_reqs] (a batch padded to a fixed capacity) get (-1, -1).
#include "mvp_internal.cuh"
#include "ptx.cuh"

namespace mvp {

namespace {

constexpr int kFillThreads = 256;

__global__ void __launch_bounds__(kFillThreads) fill_query_ranges_kernel(FillParams p) {
  // The attention call that follows may set up while this kernel runs (it
  // waits for this kernel's writes before reading the table).
  griddep_launch_dependents();
  const int t = blockIdx.x * kFillThreads + threadIdx.x;
  if (t >= p.num_tokens) return;
  if (t >= __ldg(p.qsl + p.num_reqs)) {  // a row past the batch (capacity padding)
    reinterpret_cast<int2*>(p.out)[t] = make_int2(-1, -1);
    return;
  }
  // request b with qsl[b] <= t < qsl[b + 1]; requests with q_len 0 have
  // qsl[b] == qsl[b + 1] and can never match.
  int lo = 0, hi = p.num_reqs - 1;
  while (lo < hi) {
    int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.qsl + mid) <= t) lo = mid; else hi = mid - 1;
  }
  const int b = lo;
  const int first = __ldg(p.qsl + b);
  const int q_len = __ldg(p.qsl + b + 1) - first;
  const int ctx = __ldg(p.seq_lens + b) - q_len;
  const int q_abs = ctx + (t - first);
  int rs = -1, re = -1;
  const int2* r = reinterpret_cast<const int2*>(p.ranges) + static_cast<size_t>(b) * p.max_ranges;
  for (int i = 0; i < p.max_ranges; ++i) {
    const int2 e = __ldg(r + i);
    if (e.x < e.y && e.x <= q_abs && q_abs <= e.y) {
      rs = e.x;
      re = e.y;
    }
  }
  reinterpret_cast<int2*>(p.out)[t] = make_int2(rs, re);
  if (rs >= 0 && p.rows_written) {
    // Benign race: every writer stores the same value.
    *reinterpret_cast<volatile int32_t*>(p.rows_written) = p.num_tokens;
  }
}

}  // namespace

cudaError_t launch_fill(const FillParams& p, cudaStream_t stream) {
  if (p.rows_written) {
    cudaError_t e = cudaMemsetAsync(p.rows_written, 0, sizeof(int32_t), stream);
    if (e != cudaSuccess) return e;
  }
  if (p.num_tokens <= 0) return cudaSuccess;
  const int grid = (p.num_tokens + kFillThreads - 1) / kFillThreads;
  fill_query_ranges_kernel<<<grid, kFillThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mvp
