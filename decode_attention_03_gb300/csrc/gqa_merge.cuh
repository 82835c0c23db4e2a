// Separate merge kernels: the public gqa_merge / gqa_merge_partial, the second launch of the
// tcgen05 path (and of any call with merge_mode 1) and the second pass of paged decode.
// Each folds a row's split or partition partials with the page's online-softmax merge
// (page "kernbench2 ... _gqa_attention_decode_long.py", _merge_running), then O / l.
#pragma once
#include "gqa_kernels.cuh"

namespace gqa {

// Merge kernels: W warps fold one row (W = 1 when every row has at most kMergeChunk partials,
// else 4), a block of kMergeThreads threads holds kMergeThreads / (32 W) rows.
constexpr int kMergeThreads = 256;
constexpr int kMergeChunk = 8;      // partials whose loads a warp issues before folding them

// Fold the n partials of row r (page: _merge_running; the fold order does not change the
// result beyond rounding): warp w of the row's W warps takes partials w, w + W, ... in chunks
// whose m, l and O loads are all issued first, keeping a running (M, L, O) with M in log2
// units; with W > 1 the warps' states are combined through shared memory `sm` (W * (D + 2)
// floats for this row; every thread of the block must call this once).  Lane j ends with
// O[4j .. 4j+3] (D = 128) or O[2j .. 2j+1] (D = 64) of the whole row in acc, M (log2 units)
// and L.
template <int D, int W>
__device__ __forceinline__ void fold_row(const float* m, const float* l, const float* op, int n, int64_t rows,
                                         int64_t r, int w, int lane, float* sm, float& M_out, float& L_out,
                                         float (&acc)[D / 32], int64_t n_cap, uint32_t* status) {
  constexpr int PER = D / 32;
  float M = -CUDART_INF_F, L = 0.f;
  // partial slots s < n of row r, inside the n_cap slots of `rows` rows the buffers hold
  if (n > 0 && (!idx_ok((int64_t)(n - 1) * rows + r, n_cap * rows, status) || !idx_ok(r, rows, status))) n = 0;
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  for (int s0 = w; s0 < n; s0 += W * kMergeChunk) {
    float mj[kMergeChunk], lj[kMergeChunk], oj[kMergeChunk][PER];
#pragma unroll
    for (int j = 0; j < kMergeChunk; ++j) {
      const int s = s0 + j * W;
      const bool have = s < n;
      const int64_t pr = (int64_t)(have ? s : 0) * rows + r;
      mj[j] = have ? __ldcg(m + pr) * kLog2e : -CUDART_INF_F;
      lj[j] = have ? __ldcg(l + pr) : 0.f;
      const float* src = op + pr * D + lane * PER;
      if constexpr (PER == 4) {
        const float4 v = have ? __ldcg(reinterpret_cast<const float4*>(src)) : make_float4(0.f, 0.f, 0.f, 0.f);
        oj[j][0] = v.x; oj[j][1] = v.y; oj[j][2] = v.z; oj[j][3] = v.w;
      } else {
        const float2 v = have ? __ldcg(reinterpret_cast<const float2*>(src)) : make_float2(0.f, 0.f);
        oj[j][0] = v.x; oj[j][1] = v.y;
      }
    }
    float Mc = M;
#pragma unroll
    for (int j = 0; j < kMergeChunk; ++j) Mc = fmaxf(Mc, mj[j]);
    if (Mc == -CUDART_INF_F) continue;              // all empty so far
    const float so = ptx::ex2(M - Mc);              // M = -inf -> 0
    L *= so;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] *= so;
#pragma unroll
    for (int j = 0; j < kMergeChunk; ++j) {
      const float wj = ptx::ex2(mj[j] - Mc);        // empty partials -> 0
      L += wj * lj[j];
#pragma unroll
      for (int i = 0; i < PER; ++i) acc[i] += wj * oj[j][i];
    }
    M = Mc;
  }
  if constexpr (W > 1) {
    // combine the row's warps
    float* ws = sm + w * (D + 2);
#pragma unroll
    for (int i = 0; i < PER; ++i) ws[lane * PER + i] = acc[i];
    if (lane == 0) {
      ws[D] = M;
      ws[D + 1] = L;
    }
    __syncthreads();
    float Mt = -CUDART_INF_F;
#pragma unroll
    for (int k = 0; k < W; ++k) Mt = fmaxf(Mt, sm[k * (D + 2) + D]);
    float Lt = 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) acc[i] = 0.f;
    if (Mt != -CUDART_INF_F) {
#pragma unroll
      for (int k = 0; k < W; ++k) {
        const float* wk = sm + k * (D + 2);
        const float f = ptx::ex2(wk[D] - Mt);
        Lt += f * wk[D + 1];
#pragma unroll
        for (int i = 0; i < PER; ++i) acc[i] += f * wk[lane * PER + i];
      }
    }
    M = Mt;
    L = Lt;
  }
  M_out = M;
  L_out = L;
}

// Second pass of paged decode: for every output row of a sequence with more than one
// partition, fold its partitions' partials (page: _merge_running, then O / l) into the
// 16-bit output.  W warps per row; rows of one-partition or empty sequences were written by
// the first pass.  Launched as a programmatic dependent of the partition pass: it waits for
// that grid before reading the partials.
template <int D, bool BF16, int W>
__global__ void __launch_bounds__(kMergeThreads)
gqa_paged_merge_kernel(const DecodeArgs a) {
  constexpr int PER = D / 32, RPB = kMergeThreads / (32 * W);
  __shared__ float sm[RPB][W * (D + 2)];
  if (threadIdx.x == 0) ptx::grid_launch_dependents();   // the next decode step may set up meanwhile
  ptx::grid_dependency_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rr = warp / W, w = warp % W;
  const int64_t r = (int64_t)blockIdx.x * RPB + rr;
  int n = 0;
  if (r < a.R && idx_ok(r / (a.T_q * a.h_q), a.B, a.status)) {
    const int b = (int)(r / (a.T_q * a.h_q));
    const int cap = min(a.max_blocks_per_seq * a.block_size, a.n_splits * a.partition_size);
    int len = __ldg(a.seq_lens + b);
    len = len < 0 ? 0 : (len > cap ? cap : len);
    n = (len + a.partition_size - 1) / a.partition_size;
  }
  float M, L, acc[PER];
  fold_row<D, W>(a.ws_m, a.ws_l, a.ws_o, n > 1 ? n : 0, a.R, r < a.R ? r : 0, w, lane, sm[rr], M, L, acc,
                 a.n_splits, a.status);
  if (n <= 1 || w != 0) return;
  const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
  for (int i = 0; i < PER; i += 2) Elem<BF16>::store2(a.o, r * D + lane * PER + i, acc[i] * inv, acc[i + 1] * inv);
}

// Public merge of n_parts partials laid out [n_parts][rows] and [n_parts][rows][D]
// (natural-log m).  W warps per row; a programmatic dependent of the kernel before it in the
// stream when the decode call launches it.
// `status`: the workspace status word that bounds checks report to (null for the public merge,
// which has no workspace: a check that fails there only skips the access).
template <int D, bool BF16, int W>
__global__ void __launch_bounds__(kMergeThreads)
gqa_merge_kernel(const float* __restrict__ m, const float* __restrict__ l, const float* __restrict__ op,
                 int n_parts, int64_t rows, __half* o, float* m_out, float* l_out, float* o_out, uint32_t* status) {
  constexpr int PER = D / 32, RPB = kMergeThreads / (32 * W);
  __shared__ float sm[RPB][W * (D + 2)];
  if (threadIdx.x == 0) ptx::grid_launch_dependents();   // the next decode step may set up meanwhile
  ptx::grid_dependency_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int rr = warp / W, w = warp % W;
  const int64_t r = (int64_t)blockIdx.x * RPB + rr;
  float M, L, acc[PER];
  fold_row<D, W>(m, l, op, r < rows ? n_parts : 0, rows, r < rows ? r : 0, w, lane, sm[rr], M, L, acc, n_parts,
                 status);
  if (r >= rows || w != 0) return;
  if (o != nullptr) {
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int i = 0; i < PER; i += 2) Elem<BF16>::store2(o, r * D + lane * PER + i, acc[i] * inv, acc[i + 1] * inv);
  } else {
    if (lane == 0) {
      m_out[r] = M * kLn2;
      l_out[r] = L;
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) o_out[r * D + lane * PER + i] = acc[i];
  }
}

}  // namespace gqa
