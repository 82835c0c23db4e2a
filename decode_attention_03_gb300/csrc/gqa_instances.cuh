// Compile-time configurations of the split-KV kernel and their launchers.
// A configuration is (d_head, query-row class, paged); the row class picks how
// many 8-row MMA n-tiles a consumer warp carries (NT) and how many warp
// columns share a tile (WN).
#pragma once
#include <cuda_runtime.h>

#include "gqa_kernels.cuh"

namespace gqa {

// row class -> (NT, WN): <=8 rows (1,1), <=16 (2,1), <=32 (2,2), <=64 (2,4)
constexpr int cls_nt(int cls) { return cls == 0 ? 1 : 2; }
constexpr int cls_wn(int cls) { return cls <= 1 ? 1 : (cls == 2 ? 2 : 4); }

// pipeline depth: ~96 KB of K/V stages when two CTAs fit on an SM; ~192 KB when
// one CTA per SM is all that fits anyway (merge scratch above 96 KB, or more than
// half of the register file: d_head 128 with two warp columns).  A deeper ring is not
// better where the split heuristic runs about one CTA per SM anyway: 6 x 32 KB stages took
// the 2^20-key step (19 splits) from 581-592 to 631 us on GB300.
template <int D, int NT, int WN>
constexpr int stages_for() {
  constexpr int stage = 2 * (D / 64) * kTile * 128;
  constexpr int scratch = kWK * WN * 8 * NT * (D + 6) * 4;
  constexpr bool one_per_sm = scratch > 96 * 1024 || (D == 128 && WN >= 2);
  return one_per_sm ? (192 * 1024) / stage : (96 * 1024) / stage;
}

// paged (persistent, one CTA per SM): as many stages as fit next to the merge scratch
// and the scheduler's tables in the 227 KB a CTA may use, between 2 and 8
template <int D, int NT, int WN>
constexpr int paged_stages_for() {
  using C8 = Cfg<D, NT, WN, 8>;
  constexpr int fixed = 1024 + C8::EPI_BUFS * C8::PSCRATCH_STRIDE + C8::PCTRL_BYTES;
  constexpr int n = (227 * 1024 - fixed) / C8::STAGE_BYTES;
  return n < 2 ? 2 : (n > 8 ? 8 : n);
}


// Dynamic shared memory of the split kernel over a ring of `tiles` 64-key tiles (Cfg's layout: the
// ring or the merge scratch, whichever is larger, then the barriers and flags), and for the cluster
// variant its receiving area after them.
template <int D, int NT, int WN>
constexpr int split_smem_bytes(int tiles, bool cluster) {
  using C1 = Cfg<D, NT, WN, 1>;
  const int pipe = tiles * C1::STAGE_BYTES;
  const int data = pipe > C1::SCRATCH_BYTES ? pipe : C1::SCRATCH_BYTES;
  const int ctrl = 2 * tiles * 8 + 16;
  return 1024 + data + (cluster ? ((ctrl + 15) & ~15) + ClusterRecv<C1::WROWS * WN, D>::BYTES : ctrl);
}

// Ring stages of SUB tiles: the split kernel's choice, fewer for the cluster variant where its
// receiving area would not fit beside them (64 query rows at d_head 128: 6 -> 5 stages)
template <int D, int NT, int WN, int SUB, bool CLUSTER>
constexpr int split_stages() {
  int st = stages_for<D, NT, WN>() / SUB;
  while (CLUSTER && st > 2 && split_smem_bytes<D, NT, WN>(st * SUB, true) > 227 * 1024) --st;
  return st;
}

// The deep-ring variant of the split kernel: a ring of kDeepRingBytes (4 stages of 32 KB at d_head
// 128), one CTA per SM, for grids that give every SM exactly one CTA.  Measured on GB300 (us per
// step; the heuristic's splits at two CTAs per SM on some SMs / one per SM with the deep ring),
// d_head 128, 4 rows per KV head: 8 KV heads, 2^20 keys 582.5 / 576.7-578.5 (19 splits; 3 and 5
// stages there 604.0 / 610.0); 2^17 keys 80.0 / 79.1; 2^16 keys 43.7 / 43.0; 2^15 keys 24.2 /
// 27.1 (27 tiles per split: too short); one KV head, 2^20 keys 87.1 / 86.0; two KV heads 154.0 /
// 154.3.
constexpr int kDeepRingBytes = 128 * 1024;

template <int D, int CLS, bool CAUSAL, bool BF16, bool CLUSTER = false, bool DEEP = false>
struct Inst {
  static_assert(!DEEP || (!CLUSTER && !CAUSAL), "the deep ring is a variant of the plain kernel");
  static constexpr int NT = cls_nt(CLS);
  static constexpr int WN = cls_wn(CLS);
  static constexpr int SUB = split_sub(D);
  static constexpr int STAGES = DEEP ? kDeepRingBytes / (SUB * Cfg<D, NT, WN, 1>::STAGE_BYTES)
                                     : split_stages<D, NT, WN, SUB, CLUSTER>();   // ring stages of SUB tiles
  using C = Cfg<D, NT, WN, STAGES * SUB>;
  static constexpr int SMEM = split_smem_bytes<D, NT, WN>(STAGES * SUB, CLUSTER);
  static_assert(SMEM <= 227 * 1024, "shared memory budget");
  static_assert(CLUSTER || SMEM == C::SMEM_BYTES, "the size formula follows Cfg's layout");

  // resident CTAs per SM; for the cluster variant, the number of clusters of kMaxClusterSplits CTAs
  // the GPU can hold at once is the occupancy reported (0: that cluster size cannot be scheduled)
  static cudaError_t prepare(int* occupancy) {
    auto fn = gqa_split_kernel<D, NT, WN, STAGES, SUB, CAUSAL, BF16, CLUSTER>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
    if (e != cudaSuccess) return e;
    if constexpr (!CLUSTER) {
      return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occupancy, fn, C::THREADS, SMEM);
    } else {
      e = cudaFuncSetAttribute(fn, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      cluster_config(cfg, attr, dim3(1, kMaxClusterSplits, 1), nullptr);
      return cudaOccupancyMaxActiveClusters(occupancy, fn, &cfg);
    }
  }
  // cluster variant: how many clusters of n CTAs (the n splits of a unit) the GPU holds at once,
  // after prepare() has set the kernel's attributes
  static cudaError_t max_clusters(int n, int* count) {
    if constexpr (!CLUSTER) {
      return cudaErrorInvalidValue;
    } else {
      if (n < 2 || n > kMaxClusterSplits) return cudaErrorInvalidValue;
      cudaLaunchConfig_t cfg = {};
      cudaLaunchAttribute attr[1];
      cluster_config(cfg, attr, dim3(1, (unsigned)n, 1), nullptr);
      return cudaOccupancyMaxActiveClusters(count, gqa_split_kernel<D, NT, WN, STAGES, SUB, CAUSAL, BF16, CLUSTER>,
                                            &cfg);
    }
  }
  static void cluster_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[1], dim3 grid, cudaStream_t st) {
    cfg.gridDim = grid;
    cfg.blockDim = dim3(C::THREADS, 1, 1);
    cfg.dynamicSmemBytes = SMEM;
    cfg.stream = st;
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = grid.y;   // the splits of one unit
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
  }
  static cudaError_t launch(dim3 grid, cudaStream_t st, const CUtensorMap& tk, const CUtensorMap& tv,
                            const DecodeArgs& a) {
    if constexpr (CLUSTER) {
      if (grid.y < 2 || grid.y > (unsigned)kMaxClusterSplits) return cudaErrorInvalidValue;
    }
    return launch_dependent(gqa_split_kernel<D, NT, WN, STAGES, SUB, CAUSAL, BF16, CLUSTER>, grid, C::THREADS, SMEM,
                            st, CLUSTER ? dim3(1, grid.y, 1) : dim3(1, 1, 1), tk, tv, a);
  }
};

template <int D, int CLS, int HG, bool BF16, bool VLLM>
struct PagedInst {
  static constexpr int NT = cls_nt(CLS);
  static constexpr int WN = cls_wn(CLS);
  static constexpr int STAGES = paged_stages_for<D, NT, WN>();
  using C = Cfg<D, NT, WN, STAGES>;
  static_assert(C::PSMEM_BYTES <= 227 * 1024, "shared memory budget");

  static cudaError_t prepare(int* occupancy) {
    auto fn = gqa_paged_kernel<D, NT, WN, STAGES, HG, BF16, VLLM>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::PSMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occupancy, fn, C::PTHREADS, C::PSMEM_BYTES);
  }
  static cudaError_t launch(dim3 grid, cudaStream_t st, const CUtensorMap& tk, const CUtensorMap& tv,
                            const DecodeArgs& a) {
    return launch_dependent(gqa_paged_kernel<D, NT, WN, STAGES, HG, BF16, VLLM>, grid, C::PTHREADS, C::PSMEM_BYTES,
                            st, dim3(1, 1, 1), tk, tv, a);
  }
};

// One unit (translation unit) per (kernel kind, d_head, element type).  Contiguous units:
// cls in [0, 4), variant = causal (0 / 1), or 2 = the deep-ring variant (plain units, d_head 128,
// cls 0).  Paged units (row-layout pool or vLLM cache layout): cls in [0, 4), variant = head
// group in {1, 2, 4} (2 and 4 only for cls 0 and 1).
#define GQA_DECLARE_UNIT(NAME)                                                                   \
  cudaError_t NAME##_prepare(int cls, int variant, int* occupancy);                              \
  cudaError_t NAME##_launch(int cls, int variant, dim3 grid, cudaStream_t st, const CUtensorMap& tk, \
                            const CUtensorMap& tv, const DecodeArgs& a);

// variant 2 of a contiguous unit: the deep-ring variant, row class 0 of the plain units at d_head
// 128 (elsewhere: invalid)
template <int D, bool BF, bool CL>
struct DeepCase {
  static cudaError_t prepare(int*) { return cudaErrorInvalidValue; }
  static cudaError_t max_clusters(int, int*) { return cudaErrorInvalidValue; }
  static cudaError_t launch(dim3, cudaStream_t, const CUtensorMap&, const CUtensorMap&, const DecodeArgs&) {
    return cudaErrorInvalidValue;
  }
};
template <bool BF>
struct DeepCase<128, BF, false> : Inst<128, 0, false, BF, false, true> {};

#define GQA_CONTIG_CASES(D, BF, CL, CALL)                                                        \
  if (variant == 2) return cls == 0 ? DeepCase<D, BF, CL>::CALL : cudaErrorInvalidValue;         \
  if (cls == 0) return variant ? Inst<D, 0, true, BF, CL>::CALL : Inst<D, 0, false, BF, CL>::CALL; \
  if (cls == 1) return variant ? Inst<D, 1, true, BF, CL>::CALL : Inst<D, 1, false, BF, CL>::CALL; \
  if (cls == 2) return variant ? Inst<D, 2, true, BF, CL>::CALL : Inst<D, 2, false, BF, CL>::CALL; \
  if (cls == 3) return variant ? Inst<D, 3, true, BF, CL>::CALL : Inst<D, 3, false, BF, CL>::CALL; \
  return cudaErrorInvalidValue;

// CL: the cluster variant (the splits of a unit merged through distributed shared memory)
#define GQA_DEFINE_CONTIG_UNIT(NAME, D, BF, CL)                                                  \
  cudaError_t NAME##_prepare(int cls, int variant, int* occupancy) {                             \
    GQA_CONTIG_CASES(D, BF, CL, prepare(occupancy))                                              \
  }                                                                                              \
  cudaError_t NAME##_clusters(int cls, int variant, int n, int* count) {                         \
    GQA_CONTIG_CASES(D, BF, CL, max_clusters(n, count))                                          \
  }                                                                                              \
  cudaError_t NAME##_launch(int cls, int variant, dim3 grid, cudaStream_t st, const CUtensorMap& tk, \
                            const CUtensorMap& tv, const DecodeArgs& a) {                        \
    GQA_CONTIG_CASES(D, BF, CL, launch(grid, st, tk, tv, a))                                     \
  }

#define GQA_PAGED_CASES(D, BF, VL, CALL)                                                         \
  if (cls == 0 && variant == 1) return PagedInst<D, 0, 1, BF, VL>::CALL;                         \
  if (cls == 0 && variant == 2) return PagedInst<D, 0, 2, BF, VL>::CALL;                         \
  if (cls == 0 && variant == 4) return PagedInst<D, 0, 4, BF, VL>::CALL;                         \
  if (cls == 1 && variant == 1) return PagedInst<D, 1, 1, BF, VL>::CALL;                         \
  if (cls == 1 && variant == 2) return PagedInst<D, 1, 2, BF, VL>::CALL;                         \
  if (cls == 1 && variant == 4) return PagedInst<D, 1, 4, BF, VL>::CALL;                         \
  if (cls == 2 && variant == 1) return PagedInst<D, 2, 1, BF, VL>::CALL;                         \
  if (cls == 3 && variant == 1) return PagedInst<D, 3, 1, BF, VL>::CALL;                         \
  return cudaErrorInvalidValue;

#define GQA_DEFINE_PAGED_UNIT(NAME, D, BF, VL)                                                   \
  cudaError_t NAME##_prepare(int cls, int variant, int* occupancy) {                             \
    GQA_PAGED_CASES(D, BF, VL, prepare(occupancy))                                               \
  }                                                                                              \
  cudaError_t NAME##_launch(int cls, int variant, dim3 grid, cudaStream_t st, const CUtensorMap& tk, \
                            const CUtensorMap& tv, const DecodeArgs& a) {                        \
    GQA_PAGED_CASES(D, BF, VL, launch(grid, st, tk, tv, a))                                      \
  }

GQA_DECLARE_UNIT(contig_d64)
GQA_DECLARE_UNIT(contig_d128)
GQA_DECLARE_UNIT(paged_d64)
GQA_DECLARE_UNIT(paged_d128)
GQA_DECLARE_UNIT(contig_d64_bf16)
GQA_DECLARE_UNIT(contig_d128_bf16)
GQA_DECLARE_UNIT(cluster_d64)
GQA_DECLARE_UNIT(cluster_d128)
GQA_DECLARE_UNIT(cluster_d64_bf16)
GQA_DECLARE_UNIT(cluster_d128_bf16)
// the cluster units also answer how many clusters of n CTAs the GPU holds at once
cudaError_t cluster_d64_clusters(int cls, int variant, int n, int* count);
cudaError_t cluster_d128_clusters(int cls, int variant, int n, int* count);
cudaError_t cluster_d64_bf16_clusters(int cls, int variant, int n, int* count);
cudaError_t cluster_d128_bf16_clusters(int cls, int variant, int n, int* count);
GQA_DECLARE_UNIT(paged_d64_bf16)
GQA_DECLARE_UNIT(paged_d128_bf16)
GQA_DECLARE_UNIT(paged_vllm_d64)
GQA_DECLARE_UNIT(paged_vllm_d128)
GQA_DECLARE_UNIT(paged_vllm_d64_bf16)
GQA_DECLARE_UNIT(paged_vllm_d128_bf16)

}  // namespace gqa
