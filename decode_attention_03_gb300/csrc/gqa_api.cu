// Host side of the C ABI (include/gqa_decode.h): argument validation, the
// split-count heuristic, workspace layout, TMA descriptor encoding and launches.
#include <cuda.h>
#include <cuda_runtime.h>

#include <cmath>
#include <cstdint>
#include <cstring>
#include <algorithm>
#include <mutex>

#include "../../include/gqa_decode.h"
#include "gqa_instances.cuh"
#include "gqa_merge.cuh"
#include "gqa_tc.cuh"

namespace gqa {
namespace {

constexpr int kVersion = 10000;            // 1.0.0
constexpr size_t kHeaderBytes = 256;        // status word (+ reserved)
constexpr int kMinTilesPerSplit = 1;        // a split streams at least one 64-key tile
constexpr uint64_t kDefaultTimeoutNs = 1000000000ull;
constexpr int kMaxDevices = 64;
constexpr int kTcMinRows = 16;              // automatic MMA path: tcgen05 from this many rows per KV head
// Automatic merge: the mma.sync split kernel folds 2 to kMaxClusterSplits splits in one cluster
// (distributed shared memory, one launch), more in the merge kernel, launched as a programmatic
// dependent; the tcgen05 kernel's splits always go to the merge kernel.  The last CTA of a unit
// folding the splits itself (merge_mode 2) is taken only on request: one CTA streaming a unit's
// partials is latency-bound (tcgen05, 128 rows x 19 splits = 1.26 MB: 42 us in-kernel against a
// few us for the merge kernel spread over the GPU; tiny workload, 64 splits: 16.7 vs 11.9 us),
// and with the merge kernel overlapping the decode kernel's tail it lost on small partials too.
// Measured on GB300 (us per step; last-CTA fold / cluster / merge kernel), inputs larger than L2,
// d_head 128 unless noted.  mma.sync kernel:
// 8 x 32768 keys, 4 rows, 3 splits 153.5 / 151.3 / 151.6; 8 rows 154.9 / 151.9 / 153.3; 16 rows
// 162.3 / 156.1 / 177.3; 32 rows 179.6 / 176.1 / 179.0; d_head 64, 16 rows 92.2 / 88.3 / 91.2, 64
// rows 211.2 / 186.2 / 210.1; 4 x 65536 keys (6 splits) 153.6 / 151.8 / 152.3; 16 x 16384 (2)
// 158.5 / 154.9 / 159.6; 2 x 131072 (12) 154.6 / 152.9 / 151.7; one sequence of 2^18 keys (24
// splits) 155.8 / - / 152.5, of 2^20 keys 586.9 / - / 582.5.  Where the cluster's receiving area
// costs a ring stage (64 rows at d_head 128: 510.9 / 518.9 / 509.5) or a resident CTA per SM,
// the merge kernel serves instead.  tcgen05 kernel (last-CTA fold / merge kernel): 8 x 32768 keys,
// 16 rows, 2 splits 160.7 / 159.7; 32 rows 162.7 / 160.8; 2^18 keys, 16 rows, 19 splits 158.9 /
// 155.2; 2 x 131072 keys, 16 rows, 9 splits 158.1 / 155.6; d_head 64, 8 x 32768, 16 rows 124.6 /
// 120.9; d_head 64, 2^18 keys, 32 rows, 19 splits 101.2 / 103.5 (the one shape where the fold
// in-kernel was faster).
// Automatic merge, short sweeps: where the heuristic asks for more splits than a cluster holds and
// every CTA of a 16-CTA cluster gets at most this many 64-key tiles, the unit's splits run as one
// cluster folding through distributed shared memory (one launch, no partials in global memory).
// Measured on GB300, 2 KV heads, 4 query rows, d_head 64, L2 flushed (us per step; heuristic's
// choice / merge kernel / one cluster of 16): 2048 keys 13.2 (32 splits folded by the last CTA) /
// 11.5 / 10.6; 4096 keys - / 12.2 (64 splits) / 11.0; 6144 keys 13.7 / 13.4 (95 splits) / 12.4;
// 8192 keys 13.8 / 13.8 / 12.6; 16384 keys 15.6 / 15.7 / 15.4 (and 9.0 vs 10.2 with the inputs in
// L2: there the heuristic's 95 splits stream faster).  Clusters of 12 / 8 / 4 at 4096 keys: 11.6 /
// 12.2 / 14.6.  Longer sweeps keep the splits, and the bandwidth, of the heuristic.
constexpr int kClusterMaxTilesPerSplit = 8;
// The deep-ring variant of the split kernel (kDeepRingBytes, one CTA per SM) needs at least this many
// 64-key tiles per split (measured: 54 tiles per split 1.6 % faster than the heuristic's grid, 27
// tiles 12 % slower)
constexpr int64_t kDeepMinTilesPerSplit = 48;
// Paged partitions chosen automatically (partition_size 0).  Page "muh_kernel_map.py" picks v1 --
// one pass over each whole sequence, no merge pass -- for seq_len <= 8192 and v2 with 512-token
// partitions above.  On GB300 the persistent kernel with 512-token partitions (and the merge pass
// launched as a programmatic dependent) measured at least as fast as v1 on every batch tried
// (vLLM layout, block 16, h_q 32, h_kv 8, d 128; us, v1 / v2-512: 384 seqs of 128-2048 keys
// 398 / 354; 1024 seqs 797 / 787; 2048 seqs 1618 / 1616; 512 seqs of 2048-8192 keys 1886 / 1637;
// 1024 seqs of 1024-8192 keys 3112 / 2945): a v1 item is a whole sequence, and whichever SMs take
// the longest ones finish last.  (Handing the sequences of a single pass out longest first, and a
// scheduler that claims items only as it needs them, later brought the first case to 314.5 /
// 306.5.)  So the automatic choice is v2; v1 is a partition_size of at least max_seq_len.
constexpr int kV2Partition = 512;

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

int d_index(int d) { return d == 64 ? 0 : (d == 128 ? 1 : -1); }

int row_class(int rows) {
  if (rows <= 8) return 0;
  if (rows <= 16) return 1;
  if (rows <= 32) return 2;
  if (rows <= 64) return 3;
  return -1;
}

bool aligned16(const void* p) { return p != nullptr && (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// ---------------------------------------------------------------- per-device state
struct DevState {
  bool ready = false;
  int sms = 0;
  int clusters[2][4][kMaxClusterSplits + 1] = {};   // [d index][row class][n]: clusters of n CTAs of the
                                                   // split kernel's cluster variant held at once
                                                   // (0 = not asked, -1 = none)
  int occ[2][4][13][2] = {};   // [d index][row class][kernel: see kernel_slot][bf16] resident CTAs
                               // per SM (cluster variant: clusters of kMaxClusterSplits the GPU holds),
                               // 0 = not prepared
};
std::mutex g_mu;
DevState g_dev[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Kernel selector `kind`: 0 contiguous, 1 contiguous with the causal tail, 2 / 3 the same two
// on the tcgen05 kernel (row class 0 stands for its single configuration), 4 / 5 the same two as
// the cluster variant of the split kernel (a unit's splits merged in one cluster), 6 the split
// kernel's deep-ring variant (no causal tail, row class 0, d_head 128), and for the paged kernel
// 100 + its head group (101, 102, 104) over the row-layout pool, 200 + its head group over the
// vLLM cache layout.
typedef cudaError_t (*PrepareFn)(int, int, int*);
typedef cudaError_t (*LaunchFn)(int, int, dim3, cudaStream_t, const CUtensorMap&, const CUtensorMap&,
                                const DecodeArgs&);
// [contiguous / paged / paged over the vLLM layout][d index][bf16]
const PrepareFn kPrepare[3][2][2] = {{{contig_d64_prepare, contig_d64_bf16_prepare},
                                      {contig_d128_prepare, contig_d128_bf16_prepare}},
                                     {{paged_d64_prepare, paged_d64_bf16_prepare},
                                      {paged_d128_prepare, paged_d128_bf16_prepare}},
                                     {{paged_vllm_d64_prepare, paged_vllm_d64_bf16_prepare},
                                      {paged_vllm_d128_prepare, paged_vllm_d128_bf16_prepare}}};
const LaunchFn kLaunch[3][2][2] = {{{contig_d64_launch, contig_d64_bf16_launch},
                                    {contig_d128_launch, contig_d128_bf16_launch}},
                                   {{paged_d64_launch, paged_d64_bf16_launch},
                                    {paged_d128_launch, paged_d128_bf16_launch}},
                                   {{paged_vllm_d64_launch, paged_vllm_d64_bf16_launch},
                                    {paged_vllm_d128_launch, paged_vllm_d128_bf16_launch}}};

// cluster variant of the split kernel [d index][bf16]
const PrepareFn kClusterPrepare[2][2] = {{cluster_d64_prepare, cluster_d64_bf16_prepare},
                                         {cluster_d128_prepare, cluster_d128_bf16_prepare}};
const LaunchFn kClusterLaunch[2][2] = {{cluster_d64_launch, cluster_d64_bf16_launch},
                                       {cluster_d128_launch, cluster_d128_bf16_launch}};

const PrepareFn kTcPrepare[2] = {tc_d64_prepare, tc_d128_prepare};
typedef cudaError_t (*TcLaunchFn)(int, int, dim3, cudaStream_t, const CUtensorMap&, const CUtensorMap&,
                                  const DecodeArgs&);
const TcLaunchFn kTcLaunch[2] = {tc_d64_launch, tc_d128_launch};

cudaError_t prepare_unit(int di, int cls, int kind, int bf16, int* occ) {
  if (kind == 2 || kind == 3) return kTcPrepare[di](kind - 2, bf16, occ);
  if (kind == 6) return kPrepare[0][di][bf16](0, 2, occ);
  if (kind == 4 || kind == 5) return kClusterPrepare[di][bf16](cls, kind - 4, occ);
  const int family = kind / 100;   // 0 contiguous, 1 paged, 2 paged over the vLLM layout
  return kPrepare[family][di][bf16](cls, kind - 100 * family, occ);
}

cudaError_t launch_unit(int di, int cls, int kind, int bf16, dim3 grid, cudaStream_t st, const CUtensorMap& tk,
                        const CUtensorMap& tv, const DecodeArgs& a) {
  if (kind == 2 || kind == 3) return kTcLaunch[di](kind - 2, bf16, grid, st, tk, tv, a);
  if (kind == 6) return kLaunch[0][di][bf16](0, 2, grid, st, tk, tv, a);
  if (kind == 4 || kind == 5) return kClusterLaunch[di][bf16](cls, kind - 4, grid, st, tk, tv, a);
  const int family = kind / 100;   // 0 contiguous, 1 paged, 2 paged over the vLLM layout
  return kLaunch[family][di][bf16](cls, kind - 100 * family, grid, st, tk, tv, a);
}

int kernel_slot(int kind) {
  if (kind < 2) return kind;
  if (kind < 4) return kind + 3;     // tcgen05: 5, 6
  if (kind < 100) return kind + 6;   // cluster variant: 10, 11; deep ring: 12
  const int hg_slot = (kind % 100) == 1 ? 0 : ((kind % 100) == 2 ? 1 : 2);
  return (kind < 200 ? 2 : 7) + hg_slot;   // paged: 2-4, vLLM layout: 7-9
}

// Whether the split kernel's cluster variant keeps the plain kernel's ring depth (its receiving area
// fits beside the ring), per (d index, row class)
template <int D, int CLS>
constexpr bool cluster_same_ring() {
  return Inst<D, CLS, false, false, false>::STAGES == Inst<D, CLS, false, false, true>::STAGES;
}
constexpr bool kClusterSameRing[2][4] = {
    {cluster_same_ring<64, 0>(), cluster_same_ring<64, 1>(), cluster_same_ring<64, 2>(), cluster_same_ring<64, 3>()},
    {cluster_same_ring<128, 0>(), cluster_same_ring<128, 1>(), cluster_same_ring<128, 2>(),
     cluster_same_ring<128, 3>()}};

// SM count and resident CTAs per SM of one kernel configuration on the current device
gqa_status device_info(int di, int cls, int kind, int bf16, int* sms, int* occ) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return GQA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DevState& st = g_dev[dev];
  if (!st.ready) {
    if (cudaDeviceGetAttribute(&st.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return GQA_ERR_CUDA;
    if (g_encode == nullptr) {
      void* fn = nullptr;
      cudaDriverEntryPointQueryResult q;
      if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
              cudaSuccess ||
          q != cudaDriverEntryPointSuccess || fn == nullptr)
        return GQA_ERR_CUDA;
      g_encode = reinterpret_cast<EncodeTiledFn>(fn);
    }
    st.ready = true;
  }
  int& o = st.occ[di][cls][kernel_slot(kind)][bf16];
  if (o == 0) {
    int v = 0;
    if (prepare_unit(di, cls, kind, bf16, &v) != cudaSuccess) return GQA_ERR_CUDA;
    // the cluster variant reports how many of its largest clusters fit (-1: none); others need >= 1
    if (v <= 0 && !(kind == 4 || kind == 5)) return GQA_ERR_CUDA;
    o = v > 0 ? v : -1;
  }
  *sms = st.sms;
  *occ = o;
  return GQA_OK;
}

typedef cudaError_t (*ClustersFn)(int, int, int, int*);
const ClustersFn kClusters[2][2] = {{cluster_d64_clusters, cluster_d64_bf16_clusters},
                                    {cluster_d128_clusters, cluster_d128_bf16_clusters}};

// Clusters of n CTAs of the split kernel's cluster variant (d index di, row class cls) the current
// device holds at once -- a cluster's CTAs are placed together, within one GPC, so this can be
// fewer than the resident CTAs divided by n; 0 when none fits or the query failed
int cluster_capacity(int di, int cls, int n) {
  if (n < 2 || n > kMaxClusterSplits) return 0;
  int sms = 0, c16 = 0;
  if (device_info(di, cls, 4, 0, &sms, &c16) != GQA_OK) return 0;   // prepares the variant's attributes
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return 0;
  std::lock_guard<std::mutex> lock(g_mu);
  int& c = g_dev[dev].clusters[di][cls][n];
  if (c == 0) {
    int v = 0;
    if (kClusters[di][0](cls, 0, n, &v) != cudaSuccess) v = 0;
    c = v > 0 ? v : -1;
  }
  return c > 0 ? c : 0;
}

// 3-D map over a (rows, cols) f16 / bf16 matrix seen as (64-column planes, rows, 64 columns):
// dims {64, rows, cols / 64} with strides {cols * 2 bytes, 128 bytes}.  A box of
// {64, box_rows, planes} lands in shared memory as `planes` consecutive [box_rows][64]
// arrays, rows 128 bytes with the 128-byte swizzle.
gqa_status encode_map(CUtensorMap* map, const void* base, uint64_t cols, uint64_t rows, uint32_t box_rows,
                      uint32_t planes, int bf16) {
  cuuint64_t dims[3] = {64, rows > 0 ? rows : 1, cols / 64};
  cuuint64_t strides[2] = {cols * 2, 128};
  cuuint32_t box[3] = {64, box_rows, planes};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                        const_cast<void*>(base), dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GQA_OK : GQA_ERR_CUDA;
}

// vLLM caches, one TMA box per (block, group of hg KV heads) -- a contiguous stretch of both
// caches -- moved in 128-byte rows:
//  * key cache [num_blocks, h_kv, D/8, block_size, 8] as the 4-D tensor (64 elements = 8 keys of
//    one 8-column chunk, block_size/8 key groups, D/8 chunks, num_blocks*h_kv heads); the box
//    {64, block/8, D/8, hg} lands as [chunks][keys][16 B], no swizzle;
//  * value cache [num_blocks, h_kv, D, block_size] as the 3-D tensor (64 elements, D*block/64
//    rows, num_blocks*h_kv heads); the box {64, D*block/64, hg} lands as [D rows][block keys]
//    with the 128-byte swizzle.
gqa_status encode_vllm_k(CUtensorMap* map, const void* base, uint64_t num_blocks, int h_kv, int D, int block_size,
                         uint32_t hg, int bf16) {
  cuuint64_t dims[4] = {64, (cuuint64_t)block_size / 8, (cuuint64_t)D / 8, num_blocks * (uint64_t)h_kv};
  cuuint64_t strides[3] = {128, (cuuint64_t)block_size * 16, (cuuint64_t)D * block_size * 2};
  cuuint32_t box[4] = {64, (cuuint32_t)block_size / 8, (cuuint32_t)D / 8, hg};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  if (dims[3] == 0) dims[3] = 1;
  CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GQA_OK : GQA_ERR_CUDA;
}

gqa_status encode_vllm_v(CUtensorMap* map, const void* base, uint64_t num_blocks, int h_kv, int D, int block_size,
                         uint32_t hg, int bf16) {
  const uint64_t rows = (uint64_t)D * block_size / 64;
  cuuint64_t dims[3] = {64, rows, num_blocks * (uint64_t)h_kv};
  cuuint64_t strides[2] = {128, (cuuint64_t)D * block_size * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)rows, hg};
  cuuint32_t estr[3] = {1, 1, 1};
  if (dims[2] == 0) dims[2] = 1;
  CUresult r = g_encode(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
                        const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? GQA_OK : GQA_ERR_CUDA;
}

// Split count: about 1.25 (b, g, split) CTAs per SM -- ceil(1.25 SMs / units) splits per
// unit -- with every CTA co-resident (at most the resident slots of the GPU) and each split
// at least kMinTilesPerSplit tiles long (short sweeps are latency-bound: more, shorter
// splits measured faster -- tiny workload, 4096 keys: 16 splits of 4 tiles 12.7 us, 64 of
// one tile 11.9 us with the merge kernel).  Measured on GB300 (a CTA streams at about
// 45 GB/s, bounded by its own ring, so a second CTA on some SMs adds bandwidth, while two on
// every SM split the work too finely): long context, 8 KV heads, splits 16 / 19 / 24 / 32 /
// 38 -> 610 / 591 / 586 / 603 / 597 us; 8 x 32768 keys, 64 units: 3 splits (192 CTAs) 153 us,
// 4 splits 157 us.  Prior art: page "muh_cc_dispatch.py", grid_even_share (grid =
// min(tiles, SMs x subscription), even shares of tiles).
int heuristic_splits(int64_t units, int64_t tiles, int sms, int occ, int min_tiles = kMinTilesPerSplit) {
  const int64_t slots = (int64_t)sms * occ;
  if (tiles <= 0) return 1;
  if (units >= sms) return 1;
  int64_t n = ((int64_t)sms * 5 + units * 4 - 1) / (units * 4);
  if (n > slots / units) n = slots / units;
  const int64_t cap = tiles / min_tiles;
  if (n > cap) n = cap;
  if (n < 1) n = 1;
  if (n > 65535) n = 65535;
  return (int)n;
}

struct Layout {
  size_t counters, m, l, o, total;
};

Layout ws_layout(int64_t units, int64_t n_parts, int64_t R, int D) {
  Layout L;
  L.counters = kHeaderBytes;
  size_t off = L.counters + align256((size_t)units * 4);
  if (n_parts <= 1) {
    L.m = L.l = L.o = 0;
    L.total = off;
    return L;
  }
  L.m = off;
  off += align256((size_t)(n_parts * R) * 4);
  L.l = off;
  off += align256((size_t)(n_parts * R) * 4);
  L.o = off;
  off += align256((size_t)(n_parts * R * D) * 4);
  L.total = off;
  return L;
}

gqa_options defaults() {
  gqa_options o;
  o.n_splits = 0;
  o.merge_mode = 0;
  o.timeout_us = 0;
  o.test_stall_cta = -1;
  o.paged_head_group = 0;
  o.causal = 0;
  o.bf16 = 0;
  o.mma_path = 0;
  return o;
}

struct ContigPlan {
  int di, cls, rows, n_splits;
  bool tc;                     // the tcgen05 kernel (else the mma.sync split kernel)
  bool cluster;                // the split kernel's cluster variant (merge_mode 3)
  bool deep;                   // the split kernel's deep-ring variant (kind 6)
  int64_t units, tiles, R;
  Layout lay;
};

// validation shared by the size query and the calls
// mma_path: 0 auto (tcgen05 above 64 query rows per KV head), 1 mma.sync, 2 tcgen05
gqa_status plan_contig(int B, int T_q, int64_t S_kv, int64_t s_begin, int64_t s_len, int h_q, int h_kv, int D,
                       int forced_splits, bool need_device, ContigPlan* p, int mma_path = 0, int merge_mode = 0,
                       bool causal = false) {
  if (B < 0 || T_q < 1 || h_q < 1 || h_kv < 1 || S_kv < 0 || s_begin < 0 || s_len < 0) return GQA_ERR_INVALID_ARG;
  if (s_begin + s_len > S_kv) return GQA_ERR_INVALID_ARG;
  if (h_q % h_kv != 0 || forced_splits < 0) return GQA_ERR_INVALID_ARG;
  if (B > 65535 || h_kv > 65535) return GQA_ERR_INVALID_ARG;
  if ((int64_t)B * S_kv >= (int64_t(1) << 31)) return GQA_ERR_INVALID_ARG;
  p->di = d_index(D);
  p->rows = (h_q / h_kv) * T_q;
  if (p->di < 0) return GQA_ERR_UNSUPPORTED;
  if (mma_path < 0 || mma_path > 2) return GQA_ERR_INVALID_ARG;
  const int64_t rows = (int64_t)(h_q / h_kv) * T_q;
  if (rows > kTcRows) return GQA_ERR_UNSUPPORTED;
  // automatic: the tcgen05 kernel from kTcMinRows rows (measured on GB300 at 2^18 keys, 8 KV
  // heads, d_head 128: 4-8 rows 171-173 us on mma.sync vs 175 us; 16 rows 177-179 vs 175; 32 rows
  // 193-195 vs 177; 64 rows 451 vs 179)
  // (merge_mode 3, a cluster of the split kernel, exists on the mma.sync kernel only: the automatic
  // choice takes that kernel then while it can serve the rows)
  p->tc = mma_path == 2 || (mma_path == 0 && rows >= kTcMinRows && !(merge_mode == 3 && rows <= 64));
  if (!p->tc && rows > 64) return GQA_ERR_UNSUPPORTED;
  p->cls = p->tc ? 0 : row_class(p->rows);
  p->units = (int64_t)B * h_kv;
  p->tiles = (s_len + kTile - 1) / kTile;
  p->R = (int64_t)B * T_q * h_q;
  if (forced_splits > 0) {
    int64_t n = forced_splits;
    if (n > p->tiles) n = p->tiles > 0 ? p->tiles : 1;
    if (n > 65535) n = 65535;
    p->n_splits = (int)n;
  } else if (need_device) {
    int sms = 0, occ = 0;
    gqa_status s = device_info(p->di, p->cls, p->tc ? 2 : 0, 0, &sms, &occ);
    if (s != GQA_OK) return s;
    // one-tile splits even where a stage holds two tiles (d_head 64): the latency-bound tiny
    // workload measured 12.3 us with 64 one-tile splits and the merge kernel, 13.5 us with 32
    // two-tile splits folded in-kernel
    p->n_splits = heuristic_splits(p->units, p->tiles, sms, occ);
  } else {
    p->n_splits = 1;
  }
  // the workspace holds the partials of the forced split count, or of the larger of the two kernels'
  // heuristic counts (their occupancies differ): one size query serves every MMA path and merge mode
  int ws_splits = p->n_splits;
  if (forced_splits == 0 && need_device) {
    int sms = 0, occ = 0;
    if (rows <= 64 && device_info(p->di, row_class(p->rows), 0, 0, &sms, &occ) == GQA_OK)
      ws_splits = std::max(ws_splits, heuristic_splits(p->units, p->tiles, sms, occ));
    if (device_info(p->di, 0, 2, 0, &sms, &occ) == GQA_OK)
      ws_splits = std::max(ws_splits, heuristic_splits(p->units, p->tiles, sms, occ));
  }
  p->lay = ws_layout(p->units, ws_splits, p->R, D);
  // merge_mode 3: the unit's splits form one thread-block cluster, at most kMaxClusterSplits CTAs
  p->cluster = false;
  if (merge_mode == 3) {
    if (p->tc) return GQA_ERR_UNSUPPORTED;
    if (p->n_splits > kMaxClusterSplits) p->n_splits = kMaxClusterSplits;
    p->cluster = p->n_splits > 1;
  } else if (merge_mode == 0 && !p->tc && need_device && p->n_splits > 1) {
    // automatic, mma.sync kernel: 2 to kMaxClusterSplits splits fold in one cluster where the
    // variant keeps the plain kernel's ring depth and every unit's cluster is resident at once
    // (one wave; a cluster variant with one CTA per SM holding clusters of 9, 16 units took 996 us
    // where the plain kernel takes 589, its clusters in two waves); a short sweep asking for more
    // splits runs as one cluster of kMaxClusterSplits; anything else goes to the merge kernel
    // (merge_in_kernel)
    const bool short_sweep = forced_splits == 0 && p->n_splits > kMaxClusterSplits &&
                             p->tiles <= (int64_t)kMaxClusterSplits * kClusterMaxTilesPerSplit;
    const bool holds = p->n_splits <= kMaxClusterSplits && kClusterSameRing[p->di][p->cls];
    if (short_sweep || holds) {
      const int n = short_sweep ? kMaxClusterSplits : p->n_splits;
      if (p->units <= (int64_t)cluster_capacity(p->di, p->cls, n)) {
        p->n_splits = n;
        p->cluster = true;
      }
    }
  }
  // automatic, mma.sync kernel without the causal tail, up to 8 rows at d_head 128: where the units
  // divide the SMs into more splits than a cluster holds, each long enough, one CTA per SM with the
  // deep ring (kDeepRingBytes) instead of the heuristic's splits at two CTAs on some SMs
  p->deep = false;
  if (merge_mode == 0 && forced_splits == 0 && need_device && !p->tc && !p->cluster && !causal && D == 128 &&
      p->cls == 0 && p->units > 0) {
    int sms = 0, occ = 0;
    if (device_info(p->di, 0, 6, 0, &sms, &occ) == GQA_OK && occ == 1 && sms % p->units == 0) {
      const int64_t n = sms / p->units;
      // (the workspace above holds the partials of ws_splits splits)
      if (n > kMaxClusterSplits && n <= ws_splits && p->tiles >= n * kDeepMinTilesPerSplit) {
        p->n_splits = (int)n;
        p->deep = true;
      }
    }
  }
  return GQA_OK;
}

// Launch with programmatic stream serialisation: the kernel may begin launching while the
// previous kernel in the stream finishes (it waits in griddepcontrol.wait before reading).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), unsigned grid, unsigned block, cudaStream_t st, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid, 1, 1);
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// one warp per row while a warp's first chunk of loads covers every partial, else four
int merge_warps(int n_parts) { return n_parts <= kMergeChunk ? 1 : 4; }

template <int D, bool BF16, int W>
cudaError_t merge_launch_w(const float* m, const float* l, const float* op, int n_parts, int64_t rows, __half* o,
                           float* mo, float* lo, float* oo, cudaStream_t st, uint32_t* status) {
  const int64_t rpb = kMergeThreads / (32 * W);
  const int64_t blocks = (rows + rpb - 1) / rpb;
  if (blocks > 2147483647LL) return cudaErrorInvalidValue;
  return launch_pdl(gqa_merge_kernel<D, BF16, W>, (unsigned)blocks, kMergeThreads, st, m, l, op, n_parts, rows, o,
                    mo, lo, oo, status);
}

// status: the calling decode's workspace status word (null for the public merge calls)
gqa_status merge_launch(const float* m, const float* l, const float* op, int n_parts, int64_t rows, int D,
                        __half* o, float* mo, float* lo, float* oo, cudaStream_t st, int bf16 = 0,
                        uint32_t* status = nullptr) {
  if (rows == 0) return GQA_OK;
  if (rows > 2147483647LL) return GQA_ERR_INVALID_ARG;
  const bool one = merge_warps(n_parts) == 1;
  cudaError_t e = cudaErrorInvalidValue;
#define GQA_MERGE_CASE(DD, BB)                                                                    \
  if (D == DD && bf16 == BB)                                                                      \
    e = one ? merge_launch_w<DD, BB, 1>(m, l, op, n_parts, rows, o, mo, lo, oo, st, status)       \
            : merge_launch_w<DD, BB, 4>(m, l, op, n_parts, rows, o, mo, lo, oo, st, status);
  GQA_MERGE_CASE(64, false)
  GQA_MERGE_CASE(64, true)
  GQA_MERGE_CASE(128, false)
  GQA_MERGE_CASE(128, true)
#undef GQA_MERGE_CASE
  return e == cudaSuccess ? GQA_OK : GQA_ERR_CUDA;
}

template <int D, bool BF16, int W>
cudaError_t paged_merge_launch_w(const DecodeArgs& a, cudaStream_t st) {
  const int64_t rpb = kMergeThreads / (32 * W);
  return launch_pdl(gqa_paged_merge_kernel<D, BF16, W>, (unsigned)((a.R + rpb - 1) / rpb), kMergeThreads, st, a);
}

// Whether the splits fold inside the decode launch (a cluster, or the unit's last CTA) rather than
// in the merge kernel: the cluster where plan_contig chose it (merge_mode 3, or automatic), the
// last CTA for merge_mode 2; otherwise (automatic, or merge_mode 1) the merge kernel.
bool merge_in_kernel(const ContigPlan& p, int merge_mode) { return p.cluster || merge_mode == 2; }

gqa_status decode_impl(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o, float* m_out,
                       float* l_out, float* op_out, int B, int T_q, int64_t S_kv, int64_t s_begin, int64_t s_len,
                       int h_q, int h_kv, int D, float scale, void* ws, size_t ws_bytes, void* stream,
                       const gqa_options* opt_in, bool partial) {
  const gqa_options opt = opt_in ? *opt_in : defaults();
  if (opt.merge_mode < 0 || opt.merge_mode > 3) return GQA_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
  if (!partial && S_kv < 1) return GQA_ERR_INVALID_ARG;
  ContigPlan p;
  // shape checks first: they need no device
  gqa_status s = plan_contig(B, T_q, S_kv, s_begin, s_len, h_q, h_kv, D, 1, false, &p, opt.mma_path);
  if (s != GQA_OK) return s;
  if (B == 0) return GQA_OK;
  // an empty key range (partial calls) loads no key or value: k and v may then be null (a rank
  // holding no keys), and the tensor maps are encoded over q, which is never read through them
  const bool no_keys = partial && s_len == 0;
  if (!aligned16(q) || !aligned16(ws)) return GQA_ERR_INVALID_ARG;
  if (!no_keys && (!aligned16(k) || !aligned16(v))) return GQA_ERR_INVALID_ARG;
  if (no_keys) k = v = q;
  if (partial) {
    if (!aligned16(m_out) || !aligned16(l_out) || !aligned16(op_out)) return GQA_ERR_INVALID_ARG;
  } else if (!aligned16(o)) {
    return GQA_ERR_INVALID_ARG;
  }
  s = plan_contig(B, T_q, S_kv, s_begin, s_len, h_q, h_kv, D, opt.n_splits, true, &p, opt.mma_path, opt.merge_mode,
                  opt.causal != 0);
  if (s != GQA_OK) return s;
  if (ws_bytes < p.lay.total) return GQA_ERR_WORKSPACE;
  int sms = 0, occ = 0;
  const int kind = p.deep ? 6 : (p.tc ? 2 : (p.cluster ? 4 : 0)) + (opt.causal ? 1 : 0);
  const int bf16 = opt.bf16 ? 1 : 0;
  s = device_info(p.di, p.cls, kind, bf16, &sms, &occ);
  if (s != GQA_OK) return s;

  CUtensorMap tk, tv;
  const uint64_t cols = (uint64_t)h_kv * D, nrows = (uint64_t)B * (uint64_t)S_kv;
  const uint32_t box_rows = p.tc ? kTcKeys : kTile * split_sub(D);   // keys per pipeline stage
  if ((s = encode_map(&tk, k, cols, nrows, box_rows, (uint32_t)D / 64, bf16)) != GQA_OK) return s;
  if ((s = encode_map(&tv, v, cols, nrows, box_rows, (uint32_t)D / 64, bf16)) != GQA_OK) return s;

  uint8_t* wsb = static_cast<uint8_t*>(ws);
  DecodeArgs a;
  std::memset(&a, 0, sizeof(a));
  a.q = reinterpret_cast<const __half*>(q);
  a.o = partial ? nullptr : reinterpret_cast<__half*>(o);
  a.m_out = partial ? m_out : nullptr;
  a.l_out = partial ? l_out : nullptr;
  a.o_part_out = partial ? op_out : nullptr;
  a.status = reinterpret_cast<uint32_t*>(wsb);
  a.counters = reinterpret_cast<uint32_t*>(wsb + p.lay.counters);
  if (p.n_splits > 1) {
    a.ws_m = reinterpret_cast<float*>(wsb + p.lay.m);
    a.ws_l = reinterpret_cast<float*>(wsb + p.lay.l);
    a.ws_o = reinterpret_cast<float*>(wsb + p.lay.o);
  }
  a.B = B;
  a.T_q = T_q;
  a.h_q = h_q;
  a.h_kv = h_kv;
  a.G = h_q / h_kv;
  a.rows = p.rows;
  a.R = p.R;
  a.S_kv = S_kv;
  a.s_begin = s_begin;
  a.s_len = s_len;
  a.n_splits = p.n_splits;
  a.merge_in_kernel = merge_in_kernel(p, opt.merge_mode) ? 1 : 0;
  a.causal = opt.causal ? 1 : 0;
  a.scale_log2 = scale * kLog2e;
  a.timeout_ns = opt.timeout_us ? (uint64_t)opt.timeout_us * 1000ull : kDefaultTimeoutNs;
  a.stall_cta = opt.test_stall_cta;

  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  dim3 grid((unsigned)h_kv, (unsigned)p.n_splits, (unsigned)B);
  if (launch_unit(p.di, p.cls, kind, bf16, grid, st, tk, tv, a) != cudaSuccess) return GQA_ERR_CUDA;
  if (p.n_splits > 1 && !a.merge_in_kernel) {
    return merge_launch(a.ws_m, a.ws_l, a.ws_o, p.n_splits, p.R, D, a.o, a.m_out, a.l_out, a.o_part_out, st, bf16,
                        a.status);
  }
  return GQA_OK;
}

struct PagedPlan {
  int di, cls, rows, max_parts;
  int64_t units, R;
  Layout lay;
};

// partition_size 0: automatic (kV2Partition)
gqa_status plan_paged(int N, int h_q, int h_kv, int D, int max_seq_len, int partition_size, PagedPlan* p) {
  if (partition_size == 0) partition_size = kV2Partition;
  if (N < 0 || h_q < 1 || h_kv < 1 || max_seq_len < 0 || partition_size < 0) return GQA_ERR_INVALID_ARG;
  if (h_q % h_kv != 0 || N > 65535 || h_kv > 65535) return GQA_ERR_INVALID_ARG;
  if (partition_size % kTile != 0) return GQA_ERR_INVALID_ARG;
  p->di = d_index(D);
  if (p->di < 0) return GQA_ERR_UNSUPPORTED;
  p->rows = h_q / h_kv;
  if (p->rows > 64) return GQA_ERR_UNSUPPORTED;
  p->cls = row_class(p->rows);
  const int64_t parts = ((int64_t)max_seq_len + partition_size - 1) / partition_size;
  if (parts > 65535) return GQA_ERR_INVALID_ARG;
  p->max_parts = parts > 0 ? (int)parts : 1;
  // the kernel runs on at most kPagedSeqs sequences per launch; the workspace serves one launch
  const int64_t n_launch = std::min<int64_t>(N, kPagedSeqs);
  p->units = n_launch * h_kv;
  p->R = n_launch * h_q;
  p->lay = ws_layout(p->units, p->max_parts, p->R, D);
  return GQA_OK;
}

// Head group and partition size of a paged call, and the SMs / resident CTAs of its kernel.
//  * head group: one item (and one TMA box) covers hg KV heads; larger boxes move the small
//    16-token blocks at full bandwidth.  Needs a single query column (G <= 16).
//  * partition_size 0: automatic (kV2Partition); `p` was planned with it.
gqa_status choose_paged(PagedPlan& p, int N, int h_q, int h_kv, int D, int max_seq_len, int block_size,
                        const gqa_options& opt, bool vllm, int* partition_size, int* hg_out, int* sms, int* occ) {
  // over the vLLM layout a TMA box holds whole blocks, so a tile (64 / hg keys) spans at least one
  const int hg_max = vllm ? std::min(4, 64 / block_size) : 4;
  int hg = opt.paged_head_group;
  if (hg == 0) {
    hg = p.cls <= 1 ? (h_kv % 4 == 0 ? 4 : (h_kv % 2 == 0 ? 2 : 1)) : 1;
    while (hg > hg_max) hg /= 2;
    while (h_kv % hg != 0) hg /= 2;
  }
  if (!(hg == 1 || hg == 2 || hg == 4) || h_kv % hg != 0 || (hg > 1 && p.cls > 1) || hg > hg_max)
    return GQA_ERR_INVALID_ARG;
  gqa_status s = device_info(p.di, p.cls, (vllm ? 200 : 100) + hg, opt.bf16 ? 1 : 0, sms, occ);
  if (s != GQA_OK) return s;
  if (*partition_size == 0) *partition_size = kV2Partition;
  *hg_out = hg;
  return GQA_OK;
}

// vllm: k_pool / v_pool are the vLLM caches ([blocks, h_kv, D/8, block, 8] and [blocks, h_kv, D, block])
gqa_status paged_impl(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool, const int32_t* tables,
                      const int32_t* lens, uint16_t* o, int N, int max_blocks, int num_blocks, int block_size,
                      int partition_size, int h_q, int h_kv, int D, float scale, int max_seq_len, void* ws,
                      size_t ws_bytes, void* stream, const gqa_options* opt_in, bool vllm) {
  const gqa_options opt = opt_in ? *opt_in : defaults();
  if (!std::isfinite(scale)) return GQA_ERR_INVALID_ARG;
  PagedPlan p;
  gqa_status s = plan_paged(N, h_q, h_kv, D, max_seq_len, partition_size, &p);
  if (s != GQA_OK) return s;
  if (!(block_size == 8 || block_size == 16 || block_size == 32 || block_size == 64)) return GQA_ERR_INVALID_ARG;
  // at most kMaxBoxesPerPart TMA boxes per partition; a box holds min(block_size, 16..64) rows
  if (partition_size / std::min(block_size, 16) > kMaxBoxesPerPart) return GQA_ERR_INVALID_ARG;
  if (vllm && (int64_t)num_blocks * h_kv * (D / 8) >= (int64_t(1) << 31)) return GQA_ERR_INVALID_ARG;
  if (max_blocks < 1 || num_blocks < 0) return GQA_ERR_INVALID_ARG;
  if ((int64_t)max_blocks * block_size >= (int64_t(1) << 31)) return GQA_ERR_INVALID_ARG;
  if ((int64_t)num_blocks * block_size >= (int64_t(1) << 31)) return GQA_ERR_INVALID_ARG;
  if (N == 0) return GQA_OK;
  if (!aligned16(q) || !aligned16(k_pool) || !aligned16(v_pool) || !aligned16(o) || !aligned16(ws) ||
      tables == nullptr || lens == nullptr || (reinterpret_cast<uintptr_t>(tables) & 3u) ||
      (reinterpret_cast<uintptr_t>(lens) & 3u))
    return GQA_ERR_INVALID_ARG;
  if (ws_bytes < p.lay.total) return GQA_ERR_WORKSPACE;
  int hg = 0, sms = 0, occ = 0;
  const int bf16 = opt.bf16 ? 1 : 0;
  if ((s = choose_paged(p, N, h_q, h_kv, D, max_seq_len, block_size, opt, vllm, &partition_size, &hg, &sms,
                        &occ)) != GQA_OK)
    return s;
  const int kind = (vllm ? 200 : 100) + hg;

  CUtensorMap tk, tv;
  const uint32_t box_rows = (uint32_t)std::min(block_size, 16 * (4 / hg));   // min(block, keys per tile)
  if (vllm) {
    if ((s = encode_vllm_k(&tk, k_pool, (uint64_t)num_blocks, h_kv, D, block_size, hg, bf16)) != GQA_OK) return s;
    if ((s = encode_vllm_v(&tv, v_pool, (uint64_t)num_blocks, h_kv, D, block_size, hg, bf16)) != GQA_OK) return s;
  } else {
    const uint64_t cols = (uint64_t)h_kv * D, nrows = (uint64_t)num_blocks * block_size;
    const uint32_t planes = (uint32_t)(hg * D / 64);
    if ((s = encode_map(&tk, k_pool, cols, nrows, box_rows, planes, bf16)) != GQA_OK) return s;
    if ((s = encode_map(&tv, v_pool, cols, nrows, box_rows, planes, bf16)) != GQA_OK) return s;
  }

  uint8_t* wsb = static_cast<uint8_t*>(ws);
  DecodeArgs a;
  std::memset(&a, 0, sizeof(a));
  a.status = reinterpret_cast<uint32_t*>(wsb);
  a.queue = reinterpret_cast<uint32_t*>(wsb) + 1;
  a.done = reinterpret_cast<uint32_t*>(wsb) + 2;
  a.counters = reinterpret_cast<uint32_t*>(wsb + p.lay.counters);
  if (p.max_parts > 1) {
    a.ws_m = reinterpret_cast<float*>(wsb + p.lay.m);
    a.ws_l = reinterpret_cast<float*>(wsb + p.lay.l);
    a.ws_o = reinterpret_cast<float*>(wsb + p.lay.o);
  }
  a.max_blocks_per_seq = max_blocks;
  a.num_blocks = num_blocks;
  a.block_size = block_size;
  a.partition_size = partition_size;
  a.T_q = 1;
  a.h_q = h_q;
  a.h_kv = h_kv;
  a.G = h_q / h_kv;
  a.rows = p.rows;
  a.n_splits = p.max_parts;
  a.merge_in_kernel = 1;
  a.scale_log2 = scale * kLog2e;
  a.timeout_ns = opt.timeout_us ? (uint64_t)opt.timeout_us * 1000ull : kDefaultTimeoutNs;
  a.stall_cta = opt.test_stall_cta;

  // persistent: one wave of CTAs pulling (sequence, partition, KV head) items from a queue;
  // batches beyond kPagedSeqs sequences run as consecutive launches on the same stream
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  for (int s0 = 0; s0 < N; s0 += kPagedSeqs) {
    const int n = std::min(kPagedSeqs, N - s0);
    a.q = reinterpret_cast<const __half*>(q) + (int64_t)s0 * h_q * D;
    a.o = reinterpret_cast<__half*>(o) + (int64_t)s0 * h_q * D;
    a.block_tables = tables + (int64_t)s0 * max_blocks;
    a.seq_lens = lens + s0;
    a.B = n;
    a.R = (int64_t)n * h_q;
    a.total_items = (int64_t)n * p.max_parts * (h_kv / hg);   // upper bound; the kernel counts the real ones
    const int64_t ctas = std::min<int64_t>((int64_t)sms * occ, a.total_items);
    if (launch_unit(p.di, p.cls, kind, bf16, dim3((unsigned)ctas, 1, 1), st, tk, tv, a) != cudaSuccess)
      return GQA_ERR_CUDA;
    if (p.max_parts > 1) {
      // second pass: fold the partitions of every multi-partition sequence
      const bool one = merge_warps(p.max_parts) == 1;
      cudaError_t e = cudaErrorInvalidValue;
      if (D == 64 && !bf16) e = one ? paged_merge_launch_w<64, false, 1>(a, st) : paged_merge_launch_w<64, false, 4>(a, st);
      if (D == 64 && bf16) e = one ? paged_merge_launch_w<64, true, 1>(a, st) : paged_merge_launch_w<64, true, 4>(a, st);
      if (D == 128 && !bf16)
        e = one ? paged_merge_launch_w<128, false, 1>(a, st) : paged_merge_launch_w<128, false, 4>(a, st);
      if (D == 128 && bf16) e = one ? paged_merge_launch_w<128, true, 1>(a, st) : paged_merge_launch_w<128, true, 4>(a, st);
      if (e != cudaSuccess) return GQA_ERR_CUDA;
    }
  }
  return GQA_OK;
}

}  // namespace
}  // namespace gqa

using namespace gqa;

extern "C" {

gqa_options gqa_default_options(void) { return defaults(); }

const char* gqa_status_string(int status) {
  switch (status) {
    case GQA_OK: return "ok";
    case GQA_ERR_INVALID_ARG: return "invalid argument";
    case GQA_ERR_UNSUPPORTED: return "unsupported shape (d_head must be 64 or 128, G*T_q <= 128; paged G <= 64)";
    case GQA_ERR_WORKSPACE: return "workspace too small";
    case GQA_ERR_CUDA: return "CUDA error";
    case GQA_ERR_TIMEOUT: return "a device wait timed out";
    case GQA_ERR_BOUNDS: return "a device bounds check failed (checked build)";
  }
  return "unknown status";
}

int gqa_version(void) { return kVersion; }

int gqa_build_flags(void) { return GQA_BOUNDS_CHECK ? GQA_BUILD_BOUNDS_CHECK : 0; }

int gqa_decode_num_splits(int batch, int T_q, int64_t S_kv, int h_q, int h_kv, int d_head) {
  try {
    ContigPlan p;
    if (S_kv < 1 || batch < 1) return -1;
    if (plan_contig(batch, T_q, S_kv, 0, S_kv, h_q, h_kv, d_head, 0, true, &p) != GQA_OK) return -1;
    return p.n_splits;
  } catch (...) {
    return -1;
  }
}

gqa_status gqa_decode_plan_ex(int batch, int T_q, int64_t S_kv, int h_q, int h_kv, int d_head,
                              const gqa_options* opt, int* n_splits, int* mma_path, int* launches, int* kernel,
                              int* fold) {
  try {
    const gqa_options o = opt ? *opt : defaults();
    if (S_kv < 1 || batch < 1 || o.merge_mode < 0 || o.merge_mode > 3) return GQA_ERR_INVALID_ARG;
    ContigPlan p;
    gqa_status s = plan_contig(batch, T_q, S_kv, 0, S_kv, h_q, h_kv, d_head, o.n_splits, true, &p, o.mma_path,
                               o.merge_mode, o.causal != 0);
    if (s != GQA_OK) return s;
    const bool in_kernel = merge_in_kernel(p, o.merge_mode);
    if (n_splits) *n_splits = p.n_splits;
    if (mma_path) *mma_path = p.tc ? 2 : 1;
    if (launches) *launches = (p.n_splits > 1 && !in_kernel) ? 2 : 1;
    if (kernel)
      *kernel = p.tc ? GQA_KERNEL_TCGEN05
                     : (p.cluster ? GQA_KERNEL_SPLIT_CLUSTER : (p.deep ? GQA_KERNEL_SPLIT_DEEP : GQA_KERNEL_SPLIT));
    if (fold)
      *fold = p.n_splits <= 1 ? GQA_FOLD_NONE
                              : (p.cluster ? GQA_FOLD_CLUSTER : (in_kernel ? GQA_FOLD_LAST_CTA : GQA_FOLD_MERGE_KERNEL));
    return GQA_OK;
  } catch (...) {
    return GQA_ERR_CUDA;
  }
}

gqa_status gqa_decode_plan(int batch, int T_q, int64_t S_kv, int h_q, int h_kv, int d_head, const gqa_options* opt,
                           int* n_splits, int* mma_path, int* launches) {
  return gqa_decode_plan_ex(batch, T_q, S_kv, h_q, h_kv, d_head, opt, n_splits, mma_path, launches, nullptr,
                            nullptr);
}

size_t gqa_decode_workspace_size(int batch, int T_q, int64_t S_kv, int h_q, int h_kv, int d_head, int n_splits) {
  try {
    ContigPlan p;
    if (plan_contig(batch, T_q, S_kv, 0, S_kv, h_q, h_kv, d_head, n_splits, true, &p) != GQA_OK) return 0;
    return p.lay.total;
  } catch (...) {
    return 0;
  }
}

size_t gqa_workspace_size(int batch, int T_q, int64_t S_kv, int h_q, int h_kv, int d_head) {
  return gqa_decode_workspace_size(batch, T_q, S_kv, h_q, h_kv, d_head, 0);
}

gqa_status gqa_paged_plan(int num_seqs, int h_q, int h_kv, int d_head, int block_size, int max_seq_len,
                          int partition_size, int vllm_layout, const gqa_options* opt, int* partition_out,
                          int* head_group_out, int* launches_out) {
  try {
    const gqa_options o = opt ? *opt : defaults();
    PagedPlan p;
    gqa_status s = plan_paged(num_seqs, h_q, h_kv, d_head, max_seq_len, partition_size, &p);
    if (s != GQA_OK) return s;
    if (num_seqs < 1) return GQA_ERR_INVALID_ARG;
    int part = partition_size, hg = 0, sms = 0, occ = 0;
    if (!(block_size == 8 || block_size == 16 || block_size == 32 || block_size == 64)) return GQA_ERR_INVALID_ARG;
    if ((s = choose_paged(p, num_seqs, h_q, h_kv, d_head, max_seq_len, block_size, o, vllm_layout != 0, &part, &hg,
                          &sms, &occ)) != GQA_OK)
      return s;
    const int chunks = (num_seqs + kPagedSeqs - 1) / kPagedSeqs;
    if (partition_out) *partition_out = part;
    if (head_group_out) *head_group_out = hg;
    if (launches_out) *launches_out = chunks * (p.max_parts > 1 ? 2 : 1);
    return GQA_OK;
  } catch (...) {
    return GQA_ERR_CUDA;
  }
}

size_t gqa_paged_workspace_size(int num_seqs, int h_q, int h_kv, int d_head, int max_seq_len, int partition_size) {
  PagedPlan p;
  if (plan_paged(num_seqs, h_q, h_kv, d_head, max_seq_len, partition_size, &p) != GQA_OK) return 0;
  return p.lay.total;
}

gqa_status gqa_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  if (workspace == nullptr || ws_bytes < kHeaderBytes) return GQA_ERR_INVALID_ARG;
  return cudaMemsetAsync(workspace, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
             ? GQA_OK
             : GQA_ERR_CUDA;
}

gqa_status gqa_workspace_check(void* workspace, void* stream) {
  if (workspace == nullptr) return GQA_ERR_INVALID_ARG;
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (cudaStreamSynchronize(st) != cudaSuccess) return GQA_ERR_CUDA;
  uint32_t word = 0;
  if (cudaMemcpy(&word, workspace, sizeof(word), cudaMemcpyDeviceToHost) != cudaSuccess) return GQA_ERR_CUDA;
  if (word != 0 && cudaMemset(workspace, 0, sizeof(word)) != cudaSuccess) return GQA_ERR_CUDA;
  if (word & kDevBounds) return GQA_ERR_BOUNDS;
  if (word & kDevTimeout) return GQA_ERR_TIMEOUT;
  if (word & kDevBadInput) return GQA_ERR_INVALID_ARG;
  return GQA_OK;
}

gqa_status gqa_decode_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o, int batch, int T_q,
                         int64_t S_kv, int h_q, int h_kv, int d_head, float scale, void* workspace, size_t ws_bytes,
                         void* stream, const gqa_options* opt) {
  try {
    return decode_impl(q, k, v, o, nullptr, nullptr, nullptr, batch, T_q, S_kv, 0, S_kv, h_q, h_kv, d_head, scale,
                       workspace, ws_bytes, stream, opt, false);
  } catch (...) {
    return GQA_ERR_CUDA;
  }
}

gqa_status gqa_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o, int batch, int T_q,
                      int64_t S_kv, int h_q, int h_kv, int d_head, float scale, void* workspace, size_t ws_bytes,
                      void* stream) {
  return gqa_decode_ex(q, k, v, o, batch, T_q, S_kv, h_q, h_kv, d_head, scale, workspace, ws_bytes, stream, nullptr);
}

gqa_status gqa_decode_partial_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* m, float* l,
                                 float* o_part, int batch, int T_q, int64_t S_kv, int64_t s_begin, int64_t s_len,
                                 int h_q, int h_kv, int d_head, float scale, void* workspace, size_t ws_bytes,
                                 void* stream, const gqa_options* opt) {
  try {
    return decode_impl(q, k, v, nullptr, m, l, o_part, batch, T_q, S_kv, s_begin, s_len, h_q, h_kv, d_head, scale,
                       workspace, ws_bytes, stream, opt, true);
  } catch (...) {
    return GQA_ERR_CUDA;
  }
}

gqa_status gqa_decode_partial(const uint16_t* q, const uint16_t* k, const uint16_t* v, float* m, float* l,
                              float* o_part, int batch, int T_q, int64_t S_kv, int64_t s_begin, int64_t s_len, int h_q,
                              int h_kv, int d_head, float scale, void* workspace, size_t ws_bytes, void* stream) {
  return gqa_decode_partial_ex(q, k, v, m, l, o_part, batch, T_q, S_kv, s_begin, s_len, h_q, h_kv, d_head, scale,
                               workspace, ws_bytes, stream, nullptr);
}

gqa_status gqa_merge_ex(const float* m, const float* l, const float* o_part, int n_parts, int64_t rows, int d_head,
                        uint16_t* o, void* stream, const gqa_options* opt) {
  if (n_parts < 1 || rows < 0) return GQA_ERR_INVALID_ARG;
  if (d_index(d_head) < 0) return GQA_ERR_UNSUPPORTED;
  if (rows == 0) return GQA_OK;
  if (!aligned16(m) || !aligned16(l) || !aligned16(o_part) || !aligned16(o)) return GQA_ERR_INVALID_ARG;
  return merge_launch(m, l, o_part, n_parts, rows, d_head, reinterpret_cast<__half*>(o), nullptr, nullptr, nullptr,
                      reinterpret_cast<cudaStream_t>(stream), opt != nullptr && opt->bf16 ? 1 : 0);
}

gqa_status gqa_merge(const float* m, const float* l, const float* o_part, int n_parts, int64_t rows, int d_head,
                     uint16_t* o, void* stream) {
  return gqa_merge_ex(m, l, o_part, n_parts, rows, d_head, o, stream, nullptr);
}

gqa_status gqa_merge_partial(const float* m, const float* l, const float* o_part, int n_parts, int64_t rows,
                             int d_head, float* m_out, float* l_out, float* o_out, void* stream) {
  if (n_parts < 1 || rows < 0) return GQA_ERR_INVALID_ARG;
  if (d_index(d_head) < 0) return GQA_ERR_UNSUPPORTED;
  if (rows == 0) return GQA_OK;
  if (!aligned16(m) || !aligned16(l) || !aligned16(o_part) || !aligned16(m_out) || !aligned16(l_out) ||
      !aligned16(o_out))
    return GQA_ERR_INVALID_ARG;
  return merge_launch(m, l, o_part, n_parts, rows, d_head, nullptr, m_out, l_out, o_out,
                      reinterpret_cast<cudaStream_t>(stream));
}

gqa_status gqa_decode_paged_ex(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                               const int32_t* block_tables, const int32_t* seq_lens, uint16_t* o, int num_seqs,
                               int max_blocks_per_seq, int num_blocks, int block_size, int partition_size, int h_q,
                               int h_kv, int d_head, float scale, int max_seq_len, void* workspace, size_t ws_bytes,
                               void* stream, const gqa_options* opt) {
  try {
    return paged_impl(q, k_pool, v_pool, block_tables, seq_lens, o, num_seqs, max_blocks_per_seq, num_blocks,
                      block_size, partition_size, h_q, h_kv, d_head, scale, max_seq_len, workspace, ws_bytes, stream,
                      opt, false);
  } catch (...) {
    return GQA_ERR_CUDA;
  }
}

gqa_status gqa_decode_paged(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                            const int32_t* block_tables, const int32_t* seq_lens, uint16_t* o, int num_seqs,
                            int max_blocks_per_seq, int num_blocks, int block_size, int partition_size, int h_q,
                            int h_kv, int d_head, float scale, int max_seq_len, void* workspace, size_t ws_bytes,
                            void* stream) {
  return gqa_decode_paged_ex(q, k_pool, v_pool, block_tables, seq_lens, o, num_seqs, max_blocks_per_seq, num_blocks,
                             block_size, partition_size, h_q, h_kv, d_head, scale, max_seq_len, workspace, ws_bytes,
                             stream, nullptr);
}

gqa_status gqa_decode_paged_vllm_ex(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                    const int32_t* block_tables, const int32_t* seq_lens, uint16_t* o, int num_seqs,
                                    int max_blocks_per_seq, int num_blocks, int block_size, int partition_size,
                                    int h_q, int h_kv, int d_head, float scale, int max_seq_len, void* workspace,
                                    size_t ws_bytes, void* stream, const gqa_options* opt) {
  try {
    return paged_impl(q, k_cache, v_cache, block_tables, seq_lens, o, num_seqs, max_blocks_per_seq, num_blocks,
                      block_size, partition_size, h_q, h_kv, d_head, scale, max_seq_len, workspace, ws_bytes, stream,
                      opt, true);
  } catch (...) {
    return GQA_ERR_CUDA;
  }
}

gqa_status gqa_decode_paged_vllm(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                 const int32_t* block_tables, const int32_t* seq_lens, uint16_t* o, int num_seqs,
                                 int max_blocks_per_seq, int num_blocks, int block_size, int partition_size, int h_q,
                                 int h_kv, int d_head, float scale, int max_seq_len, void* workspace,
                                 size_t ws_bytes, void* stream) {
  return gqa_decode_paged_vllm_ex(q, k_cache, v_cache, block_tables, seq_lens, o, num_seqs, max_blocks_per_seq,
                                  num_blocks, block_size, partition_size, h_q, h_kv, d_head, scale, max_seq_len,
                                  workspace, ws_bytes, stream, nullptr);
}

}  // extern "C"
