// Range-table fill on the GPU.
//
// Restates vLLM PR #50294 review, "Key source snippets",
// fill_mm_prefix_query_ranges, as a data-parallel integer kernel: every
// packed query row t of request b gets the closed (start, end) of the last
// listed valid (start < end) range of b that holds the row's absolute
// position ctx + (t - query_start_loc[b]), or (-1, -1) -- exactly the row the
// page's span writes leave behind, since later spans overwrite earlier ones
// and a span covers precisely the rows whose position lies in [start, end]
// within the scheduled chunk.  Every row [0, num_tokens) is written (unlike
// the page, which leaves the buffer untouched when nothing is covered), and
// rows_written receives the page's return value.  Rows at or past
// query_start_loc[num_reqs] (a batch padded to a fixed capacity) get (-1, -1).
//
// A CTA covers 1024 consecutive rows (four per thread).  When they belong to
// a few requests (the prefill case) the CTA restates the page's span
// procedure: each valid range of those requests marks the rows of its span,
// clipped to the CTA's rows, in a shared row -> range map with atomicMax over
// the range's position in the list (the lanes of a warp mark a span's rows
// together), so the last listed range wins as in the page's write order;
// then every thread stores its rows.  That is O(rows + ranges) work with each range read once per
// CTA.  Otherwise (many short requests, e.g. decode rows) each row finds its
// request by binary search and scans that request's ranges in list order.
#include <climits>

#include "mvp_internal.cuh"
#include "ptx.cuh"

namespace mvp {

namespace {

constexpr int kFillThreads = 256;
constexpr int kRowsPerThread = 4;
constexpr int kFillRows = kFillThreads * kRowsPerThread;  // rows of one CTA
// The span procedure runs when the CTA's requests have at most this many
// ranges between them (eight per thread).
constexpr int kMaxSpanRanges = 8 * kFillThreads;

// Request b with qsl[b] <= t < qsl[b + 1] (requests with q_len 0 have
// qsl[b] == qsl[b + 1] and never match).
__device__ __forceinline__ int request_of(const FillParams& p, int t) {
  int lo = 0, hi = p.num_reqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (__ldg(p.qsl + mid) <= t) lo = mid; else hi = mid - 1;
  }
  return lo;
}

// Warp-collective form for one row t: a 32-ary search, each step probing 32
// evenly spaced offsets (3 steps for 4096 requests instead of 12 dependent
// loads).  The answer is the largest b with qsl[b] <= t.
__device__ __forceinline__ int request_of_warp(const FillParams& p, int t, int lane) {
  int lo = 0, n = p.num_reqs;  // the answer lies in [lo, lo + n)
  while (n > 1) {
    const int c = lo + static_cast<int>(static_cast<long long>(lane) * n / 32);
    const unsigned m = __ballot_sync(0xffffffffu, __ldg(p.qsl + c) <= t);  // a prefix of the lanes
    const int k = m != 0u ? 31 - __clz(m) : 0;
    const int next = k == 31 ? lo + n : lo + static_cast<int>(static_cast<long long>(k + 1) * n / 32);
    lo += static_cast<int>(static_cast<long long>(k) * n / 32);
    n = next - lo;
  }
  return lo;
}

__global__ void __launch_bounds__(kFillThreads) fill_query_ranges_kernel(FillParams p) {
  // The attention call that follows may set up while this kernel runs (it
  // waits for this kernel's writes before reading the table).
  griddep_launch_dependents();
  __shared__ int s_idx[kFillRows];  // per row: flat index b * max_ranges + i of its range, or -1
  __shared__ int s_req[2];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t0 = blockIdx.x * kFillRows;
  const int n_batch = min(__ldg(p.qsl + p.num_reqs), p.num_tokens);  // rows that belong to a request
  const int t_last = min(t0 + kFillRows, n_batch) - 1;               // this CTA's last such row
  if (warp < 2) {
    // warp 0: the request of the CTA's first row; warp 1: of its last row
    const int b = t0 <= t_last ? request_of_warp(p, warp == 0 ? t0 : t_last, lane) : -1;
    if (lane == 0) s_req[warp] = b;
  }
#pragma unroll
  for (int k = 0; k < kRowsPerThread; ++k) s_idx[threadIdx.x + k * kFillThreads] = -1;
  __syncthreads();
  const int b0 = s_req[0], b1 = s_req[1];
  const int2* rng = reinterpret_cast<const int2*>(p.ranges);
  const bool spans = b0 >= 0 && static_cast<long long>(b1 - b0 + 1) * p.max_ranges <= kMaxSpanRanges &&
                     static_cast<long long>(b1 + 1) * p.max_ranges <= INT_MAX;  // flat indices fit an int
  if (spans) {
    // The span procedure over the CTA's rows [t0, t_last]: pair j is range
    // j % max_ranges of request b0 + j / max_ranges.  Each thread reads the
    // pairs j = m * 256 + lane * 8 + warp (so every warp gets an eighth of
    // them) and clips their spans; then each warp marks its lanes' spans
    // with all 32 lanes, one row per lane per round.
    const int n_pairs = (b1 - b0 + 1) * p.max_ranges;
    for (int base = 0; base < n_pairs; base += kFillThreads) {
      const int j = base + lane * 8 + warp;
      long long lo = 1, hi = 0;  // empty
      if (j < n_pairs) {
        const int b = b0 + j / p.max_ranges;
        const int2 e = __ldg(rng + static_cast<size_t>(b0) * p.max_ranges + j);
        if (e.x < e.y) {  // degenerate ranges are skipped
          const int first = __ldg(p.qsl + b);
          const int q_len = __ldg(p.qsl + b + 1) - first;
          const long long ctx = static_cast<long long>(__ldg(p.seq_lens + b)) - q_len;
          // packed rows of the span: first + clip([start - ctx, end - ctx], [0, q_len - 1]), within the CTA
          lo = max(first + max(static_cast<long long>(e.x) - ctx, 0LL), static_cast<long long>(t0));
          hi = min(first + min(static_cast<long long>(e.y) - ctx, q_len - 1LL), static_cast<long long>(t_last));
        }
      }
      const int flat = static_cast<int>(static_cast<long long>(b0) * p.max_ranges + j);
      // rows relative to t0 (0..kFillRows-1 when not empty)
      const int rlo = lo <= hi ? static_cast<int>(lo - t0) : 1;
      const int rhi = lo <= hi ? static_cast<int>(hi - t0) : 0;
      unsigned todo = __ballot_sync(0xffffffffu, rlo <= rhi);
      while (todo != 0u) {
        const int k = __ffs(todo) - 1;
        todo &= todo - 1u;
        const int klo = __shfl_sync(0xffffffffu, rlo, k);
        const int khi = __shfl_sync(0xffffffffu, rhi, k);
        const int kflat = __shfl_sync(0xffffffffu, flat, k);
        for (int row = klo + lane; row <= khi; row += 32) atomicMax(&s_idx[row], kflat);
      }
    }
    __syncthreads();
  }
  bool hit = false;
#pragma unroll
  for (int k = 0; k < kRowsPerThread; ++k) {
    const int t = t0 + threadIdx.x + k * kFillThreads;
    int rs = -1, re = -1;
    if (t <= t_last) {
      if (spans) {
        const int i = s_idx[t - t0];
        if (i >= 0) {
          const int2 e = __ldg(rng + i);
          rs = e.x;
          re = e.y;
        }
      } else {
        // Rows of many requests: scan the row's request in list order.
        const int b = request_of(p, t);
        const int first = __ldg(p.qsl + b);
        const int q_len = __ldg(p.qsl + b + 1) - first;
        const int q_abs = __ldg(p.seq_lens + b) - q_len + (t - first);
        const int2* r = rng + static_cast<size_t>(b) * p.max_ranges;
        for (int i = 0; i < p.max_ranges; ++i) {
          const int2 e = __ldg(r + i);
          if (e.x < e.y && e.x <= q_abs && q_abs <= e.y) {
            rs = e.x;
            re = e.y;
          }
        }
      }
    }
    if (t < p.num_tokens) reinterpret_cast<int2*>(p.out)[t] = make_int2(rs, re);
    hit = hit || rs >= 0;
  }
  if (__syncthreads_or(hit) && threadIdx.x == 0 && p.rows_written) {
    // Benign race between CTAs: every writer stores the same value.
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
  const int grid = static_cast<int>((static_cast<long long>(p.num_tokens) + kFillRows - 1) / kFillRows);
  fill_query_ranges_kernel<<<grid, kFillThreads, 0, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace mvp
