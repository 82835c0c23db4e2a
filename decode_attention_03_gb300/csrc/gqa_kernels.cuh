// Split-KV GQA decode kernels for sm_103a.
//
// Work unit: one (sequence b, KV head g) pair -- the G*T_q query rows that share KV
// head g -- against one contiguous slice of the key axis.  Page "kernbench2 ...
// _gqa_attention_decode_long.py" ("GQA fused-attention decode kernel -- long
// context") describes the same decomposition for a PE mesh: every rank sweeps its
// S_kv slice in tiles, keeps a running (m, l, O) and partials are merged with
// _merge_running; here the ranks become CTAs and the reduce-to-root becomes the
// last-arriving CTA of the unit merging all slices.  The paged variant follows page
// "muh_kernel_map.py", VLLM_KERNEL_MAP 'paged_attention_v2' (a pass per 512-token
// partition, then a cross-partition merge).
//
// CTA layout: kWK*WN consumer warps + 1 producer warp.
// Q, K, V and O are f16 or bf16 (one instantiation each); scores, softmax statistics,
// partials and accumulation are fp32.
//
//  * producer: TMA 3-D tensor loads (64 columns x rows x the head's 64-column
//    planes, 128-byte swizzle) of each 64-key K and V tile into a STAGES-deep ring of
//    shared-memory buffers, signalled through mbarriers (full / empty).  One box
//    covers the whole tile (contiguous) or one KV block (paged).
//  * consumer warp (ks, nc): keys [16*ks, 16*ks+16) of every tile, query n-tiles
//    [nc*NT, nc*NT+NT) (8 query rows each).  Scores are computed transposed,
//    S^T = K Q^T (keys on the MMA's M side, so G*T_q = 4 wastes only half of an n=8
//    tile), the softmax runs in the accumulator layout, P is transposed in registers
//    (movmatrix) into the B operand of O^T += V^T P^T.  Each warp keeps its own
//    running (m, l, O) over its keys; the warps' states are merged through shared
//    memory at the end of the slice.
//
// gqa_split_kernel: one CTA per (KV head, split, sequence) of a contiguous K/V (CAUSAL:
//   the speculative-verification tail mask, a separate instantiation).
// gqa_paged_kernel: persistent, one CTA per SM; a scheduler warp takes
//   (sequence, partition, KV head) items from an atomic queue and reads the
//   partition's block ids ahead of time, the producer warp streams the items'
//   tiles through one ring that runs across items, so a partition's ramp-up
//   overlaps the previous one's tail.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <math_constants.h>
#include <stdint.h>

#include "ptx.cuh"

namespace gqa {

constexpr int kWK = 4;             // consumer warps along the key axis
constexpr int kTile = 16 * kWK;    // keys per pipeline stage
constexpr uint32_t kDevTimeout = 1u;
constexpr uint32_t kDevBadInput = 2u;
constexpr uint32_t kDevBounds = 4u;     // a bounds check failed (checked build only)
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxBoxesPerPart = 1024;  // paged: TMA boxes (blocks or block slices) of one partition
// paged kernel: descriptors in flight between scheduler and workers.  Two (the producer's item and
// the next) keep the TMA ring fed across items and bound the work a CTA has claimed ahead; with
// four, and the next item claimed before a slot was free, 384 sequences of 128-2048 keys in one
// partition each took 368.9 instead of 337.5 us on GB300 (the same in 512-key partitions: 312.9
// instead of 306.8 us; 64 sequences of 1024-16384 keys: 333.0 instead of 331.9 us)
constexpr int kItemSlots = 2;
constexpr int kPagedSeqs = 1024;   // paged kernel: sequences per launch (the host splits larger batches)
constexpr int kSizeClasses = 64;   // paged kernel, single pass: length classes of the longest-first order

struct DecodeArgs {
  const __half* q;        // (B, T_q, h_q*D)
  __half* o;              // (B, T_q, h_q*D) final output, or null
  float* m_out;           // partial output (natural-log max), rows (b, t, h), or null
  float* l_out;
  float* o_part_out;      // (rows, D) unnormalised
  float* ws_m;            // split partials [n_splits][R]
  float* ws_l;
  float* ws_o;            // [n_splits][R][D]
  uint32_t* status;       // device error bits
  uint32_t* counters;     // one arrival counter per (b, g) unit
  uint32_t* queue;        // paged: next work item
  uint32_t* done;         // paged: CTAs finished (the last one resets queue and done)
  // paged
  const int32_t* block_tables;
  const int32_t* seq_lens;
  int max_blocks_per_seq;
  int num_blocks;
  int block_size;
  int partition_size;
  int64_t total_items;    // paged: num_seqs * max_parts * h_kv
  // shape
  int B, T_q, h_q, h_kv, G, rows;  // rows = G*T_q query rows per unit
  int64_t R;                        // B*T_q*h_q rows of the output
  int64_t S_kv;                     // contiguous: keys per sequence
  int64_t s_begin, s_len;           // contiguous: key range swept
  int n_splits;                     // contiguous: splits per unit; paged: max partitions per sequence
  int merge_in_kernel;              // last CTA of a unit merges the splits
  int causal;                       // query token t sees keys j <= S_kv - T_q + t only
  float scale_log2;                 // scale * log2(e)
  uint64_t timeout_ns;
  int stall_cta;                    // test hook (-1 none): contiguous, the CTA whose producer withholds
                                    // its second tile; paged, the queue item whose second tile is withheld
};

template <int D, int NT, int WN, int STAGES>
struct Cfg {
  static constexpr int HALVES = D / 64;
  static constexpr int KV_BYTES = HALVES * kTile * 128; // one K (or V) tile: kTile rows x D f16
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int CONSUMERS = kWK * WN;
  static constexpr int CTHREADS = CONSUMERS * 32;
  static constexpr int THREADS = (CONSUMERS + 1) * 32;
  static constexpr int WROWS = 8 * NT;                   // query rows per consumer warp
  static constexpr int OSTRIDE = D + 4;                  // padded row of the merge scratch
  static constexpr int WSCRATCH = WROWS * (OSTRIDE + 2); // floats per warp
  static constexpr int SCRATCH_BYTES = CONSUMERS * WSCRATCH * 4;
  static constexpr int PIPE_BYTES = STAGES * STAGE_BYTES;
  // split kernel: the merge scratch reuses the drained ring
  static constexpr int DATA_BYTES = PIPE_BYTES > SCRATCH_BYTES ? PIPE_BYTES : SCRATCH_BYTES;
  static constexpr int CTRL_BYTES = 2 * STAGES * 8 + 16;
  static constexpr int SMEM_BYTES = 1024 + DATA_BYTES + CTRL_BYTES;
  // paged kernel: the ring stays busy across items, so the scratch has its own space,
  // double-buffered between the consumers and the epilogue warp
  // (a single buffer when two would crowd out the ring: many query rows per KV head)
  static constexpr int PSCRATCH_STRIDE = (SCRATCH_BYTES + 1023) & ~1023;
  static constexpr int EPI_BUFS = 2 * PSCRATCH_STRIDE <= 48 * 1024 ? 2 : 1;
  static constexpr int PSCRATCH_OFF = PIPE_BYTES;
  static constexpr int PCTRL_OFF = PIPE_BYTES + EPI_BUFS * PSCRATCH_STRIDE;
  static constexpr int PCTRL_BYTES = (2 * STAGES + 2 * kItemSlots + 2 * EPI_BUFS) * 8 + 16 +
                                     (kItemSlots + EPI_BUFS) * 48 + kItemSlots * kMaxBoxesPerPart * 4 +
                                     (3 * kPagedSeqs + 1 + kSizeClasses) * 4;
  static constexpr int PSMEM_BYTES = 1024 + PCTRL_OFF + PCTRL_BYTES;
  static constexpr int PTHREADS = (CONSUMERS + 3) * 32;          // + producer, scheduler, epilogue
};

// ---- opt-in bounds checks.  Built with -DGQA_BOUNDS_CHECK=1 (the checked library), every
// computed global-memory index and shared-memory address of the kernels is compared with the
// extent of the buffer or shared-memory region it falls in before the access; one out of range
// sets kDevBounds in the status word (when there is one) and the access is skipped, or made at
// the region's first address where a warp-collective instruction must still execute -- nothing
// traps.  In the regular build every check is the constant true.
#ifndef GQA_BOUNDS_CHECK
#define GQA_BOUNDS_CHECK 0
#endif

// 0 <= i < n
__device__ __forceinline__ bool idx_ok(int64_t i, int64_t n, uint32_t* status) {
#if GQA_BOUNDS_CHECK
  if (i < 0 || i >= n) {
    if (status != nullptr) atomicOr(status, kDevBounds);
    return false;
  }
#endif
  return true;
}

// [addr, addr + bytes) inside the shared-memory region [lo, hi)
__device__ __forceinline__ bool smem_ok(uint32_t addr, uint32_t bytes, uint32_t lo, uint32_t hi, uint32_t* status) {
#if GQA_BOUNDS_CHECK
  if (addr < lo || addr + bytes > hi) {
    if (status != nullptr) atomicOr(status, kDevBounds);
    return false;
  }
#endif
  return true;
}

// an address for a warp-collective shared-memory read: `addr` when in range, else `lo`
__device__ __forceinline__ uint32_t smem_clamp(uint32_t addr, uint32_t bytes, uint32_t lo, uint32_t hi,
                                               uint32_t* status) {
  return smem_ok(addr, bytes, lo, hi, status) ? addr : lo;
}

// A shared-memory region [lo, hi) and the status word its checks report to.
struct Win {
  uint32_t lo, hi;
  uint32_t* status;
};

// Row r of a unit (0 <= r < G*T_q) is query token r / G, head g*G + r % G.
__device__ __forceinline__ int64_t out_row(const DecodeArgs& a, int b, int g, int r) {
  const int tq = r / a.G, hh = r - tq * a.G;
  return ((int64_t)b * a.T_q + tq) * a.h_q + (int64_t)g * a.G + hh;
}

// Shared-memory tile layout.  A K (or V) tile arrives as consecutive TMA boxes of
// `rb` rows (the whole tile for contiguous K/V, a KV block -- or part of one -- when
// paged); a box holds BOXP planes [rb][64]: the 64-column slices of the tile's heads
// (D/64 per head, heads one after the other), each row of a plane 128 bytes with its
// 16-byte chunks swizzled (chunk ^ row % 8).  Offset of `row` within the tile, before
// the plane and chunk terms:
template <int BOXP>
__device__ __forceinline__ int row_offset(int row, int rb) {
  return (row / rb) * (rb * 128 * BOXP) + (row % rb) * 128;
}

// address of 16-byte chunk c (of D/8) of `row`, given row_offset(row); planes rb*128 bytes apart
__device__ __forceinline__ uint32_t chunk_addr(uint32_t base, int row_off, int row, int c, int plane_bytes) {
  return base + row_off + (c >> 3) * plane_bytes + ((((c & 7) ^ (row & 7))) << 4);
}

__device__ __forceinline__ void raise_timeout(const DecodeArgs& a, volatile int* flags) {
  atomicOr(a.status, kDevTimeout);
  flags[0] = 1;
}

// Element type of Q, K, V and O: IEEE binary16 (BF16 = false) or bfloat16.  The MMA
// consumes the raw 16-bit values; only the MMA kind, the packing of P and the output
// rounding depend on the type.
template <bool BF16>
struct Elem {
  static __device__ __forceinline__ void mma(float (&d)[4], const uint32_t (&a)[4], const uint32_t (&b)[2]) {
    if constexpr (BF16) ptx::mma_16816_bf16(d, a, b); else ptx::mma_16816(d, a, b);
  }
  static __device__ __forceinline__ uint32_t pack(float lo, float hi) {
    if constexpr (BF16) return ptx::pack_bf162(lo, hi); else return ptx::pack_half2(lo, hi);
  }
  static __device__ __forceinline__ void store(__half* base, int64_t i, float x) {
    if constexpr (BF16) {
      reinterpret_cast<__nv_bfloat16*>(base)[i] = __float2bfloat16_rn(x);
    } else {
      base[i] = __float2half_rn(x);
    }
  }
  static __device__ __forceinline__ void store2(__half* base, int64_t i, float lo, float hi) {
    reinterpret_cast<uint32_t*>(base + i)[0] = pack(lo, hi);
  }
};

// =====================================================================================
// consumer warp state and per-tile math
// =====================================================================================
template <int D, int NT>
struct WarpState {
  static constexpr int KD = D / 16;   // k-steps over d (QK) / m-tiles over d (PV)
  uint32_t qf[NT][KD][2];             // Q^T fragments (B operand of S^T = K Q^T)
  float acc[KD][NT][4];               // O^T accumulators (rows d, columns query rows)
  float m_run[NT][2];                 // running max (log2 domain), query rows 2*tq4, 2*tq4+1
  float l_run[NT][2];                 // running sum over this lane's keys
  int lim[NT][2];                     // last key index those rows may see (causal tail), else INT_MAX
};

// Q^T fragments: b0 = Q[row gq][16kk + 2tq4 ..+1], b1 = the same 8 columns further
template <int D, int NT>
__device__ __forceinline__ void load_q(WarpState<D, NT>& st, const DecodeArgs& a, int b, int g, int nc, int lane) {
  const int gq = lane >> 2, tq4 = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      // rows of the score fragment held by this lane: 2*tq4 + j of n-tile nt (token r / G)
      const int r = (nc * NT + nt) * 8 + 2 * tq4 + j;
      st.lim[nt][j] = a.causal ? (int)(a.S_kv - a.T_q + r / a.G) : 0x7fffffff;
    }
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int r = (nc * NT + nt) * 8 + gq;
    if (r < a.rows && idx_ok(out_row(a, b, g, r), a.R, a.status)) {   // the row's D elements
      const uint32_t* qp = reinterpret_cast<const uint32_t*>(a.q + out_row(a, b, g, r) * D);
#pragma unroll
      for (int kk = 0; kk < WarpState<D, NT>::KD; ++kk) {
        st.qf[nt][kk][0] = __ldg(qp + kk * 8 + tq4);
        st.qf[nt][kk][1] = __ldg(qp + kk * 8 + 4 + tq4);
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < WarpState<D, NT>::KD; ++kk) st.qf[nt][kk][0] = st.qf[nt][kk][1] = 0u;
    }
  }
}

template <int D, int NT>
__device__ __forceinline__ void reset_state(WarpState<D, NT>& st) {
#pragma unroll
  for (int i = 0; i < WarpState<D, NT>::KD; ++i)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) st.acc[i][nt][c] = 0.f;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    st.m_run[nt][0] = st.m_run[nt][1] = -CUDART_INF_F;
    st.l_run[nt][0] = st.l_run[nt][1] = 0.f;
  }
}

// Keys of this warp's slice past the range: zero their V rows so that 0 * (stale or
// NaN) cannot reach O.  The rows were written by TMA; the fence orders these generic
// writes before the next asynchronous (TMA) write into the same buffer.
// `vhead` points at the first plane of this warp's head.
template <int HALVES, int BOXP>
__device__ __forceinline__ void zero_masked_v(uint8_t* vhead, int ks, int valid, int lane, int rb, const Win& ring) {
  const int per_row = 8 * HALVES;                      // 16-byte chunks of one row of the head
  for (int i = lane; i < (16 - valid) * per_row; i += 32) {
    const int row = ks * 16 + valid + i / per_row;
    const int rem = i % per_row;
    const int off = row_offset<BOXP>(row, rb) + (rem >> 3) * (rb * 128) + (rem & 7) * 16;
    if (smem_ok(ptx::smem_u32(vhead + off), 16, ring.lo, ring.hi, ring.status))
      *reinterpret_cast<uint4*>(vhead + off) = make_uint4(0u, 0u, 0u, 0u);
  }
  ptx::fence_proxy_async_smem();
  __syncwarp();
}

// vLLM cache layout (page "muh_kernel_map.py", paged_attention_v1 key_cache
// [num_blocks, num_kv_heads, head_dim/x, block_size, x], x = 8 16-bit elements; value cache
// [num_blocks, num_kv_heads, head_dim, block_size]).  A TMA box holds one whole block
// (rb = block_size keys) of HG heads -- a contiguous stretch of each cache -- and lands as:
//  * K: [HG*D/8 chunks][rb keys][16 bytes] -- chunk-major, no swizzle: the 8 keys of an
//    ldmatrix row group are 128 consecutive bytes;
//  * V: [HG*D rows][rb keys] (V transposed), moved as 128-byte rows with the 128-byte
//    swizzle, so that the 8 d rows an ldmatrix reads hit distinct banks for every block size.
// Byte offset of element (d row, key kb) of a V box, swizzle applied:
__device__ __forceinline__ int vllm_v_offset(int drow, int kb, int rb) {
  const int off = (drow * rb + kb) * 2;
  return off ^ (((off >> 7) & 7) << 4);
}

// Keys of this warp's slice past the range, vLLM layout: zero their V columns (every d row of
// the warp's head) so that 0 * (stale or NaN) cannot reach O.  `vhead` points at the first
// row of this warp's head in the tile's first box; boxes of rb keys are box_bytes apart.
template <int D>
__device__ __forceinline__ void zero_masked_v_vllm(uint8_t* vhead, int ks, int valid, int lane, int rb,
                                                   int box_bytes, const Win& ring) {
  const int nmask = 16 - valid;
  for (int i = lane; i < D * nmask; i += 32) {
    const int drow = i / nmask;
    const int key = ks * 16 + valid + (i - drow * nmask);
    uint8_t* dst = vhead + (key / rb) * box_bytes + vllm_v_offset(drow, key % rb, rb);
    if (smem_ok(ptx::smem_u32(dst), 2, ring.lo, ring.hi, ring.status)) *reinterpret_cast<uint16_t*>(dst) = 0;
  }
  ptx::fence_proxy_async_smem();
  __syncwarp();
}

// One tile: this warp's 16 keys against its 8*NT query rows; kbase / vbase point at
// the first plane (row layout) or first chunk / d row (VLLM) of the warp's head.
template <int D, int NT, int BOXP, bool CAUSAL = false, bool BF16 = false, bool VLLM = false>
__device__ __forceinline__ void consume_tile(WarpState<D, NT>& st, uint32_t kbase, uint32_t vbase, int valid,
                                             int key0, int ks, int lane, float scale_log2, int rb, const Win& ring) {
  constexpr int KD = WarpState<D, NT>::KD;
  const int gq = lane >> 2;
  const int k_row = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int k_c0 = lane >> 4;
  const int v_row = ks * 16 + (lane & 7) + ((lane >> 4) & 1) * 8;
  const int v_c0 = (lane >> 3) & 1;
  const int k_off = row_offset<BOXP>(k_row, rb), v_off = row_offset<BOXP>(v_row, rb);
  const int plane = rb * 128;
  // VLLM: box of this lane's K row and of its V key group (keys ks*16 + 8*(lane >> 4) ..+7)
  const int box_bytes = rb * 128 * BOXP;
  const uint32_t kvb = kbase + (k_row / rb) * box_bytes + (k_row % rb) * 16;
  const int v_key = ks * 16 + (lane >> 4) * 8;
  const uint32_t vvb = vbase + (v_key / rb) * box_bytes;
  const int v_kb = v_key % rb;
  const int v_dr = (lane & 7) + ((lane >> 3) & 1) * 8;

  // ---- S^T = K Q^T : 16 keys x 8*NT query rows, fp32
  float sc[NT][4];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < KD; ++kk) {
    uint32_t af[4];
    if constexpr (VLLM) {
      ptx::ldmatrix_x4(af, smem_clamp(kvb + (kk * 2 + k_c0) * rb * 16, 16, ring.lo, ring.hi, ring.status));
    } else {
      ptx::ldmatrix_x4(af, smem_clamp(chunk_addr(kbase, k_off, k_row, kk * 2 + k_c0, plane), 16, ring.lo, ring.hi,
                                      ring.status));
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) Elem<BF16>::mma(sc[nt], af, st.qf[nt][kk]);
  }
  // ---- scale (log2 domain), mask, online softmax.  sc[nt][c]: key gq (c<2) or gq+8,
  //      query row 2*tq4 + (c&1) of n-tile nt
  float alpha[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    if constexpr (CAUSAL) {
      // last key of the slice each of this lane's two rows may see (range end, causal tail)
      const int last0 = min(valid - 1, st.lim[nt][0] - key0);
      const int last1 = min(valid - 1, st.lim[nt][1] - key0);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int key = gq + ((c >> 1) << 3);
        sc[nt][c] = key <= ((c & 1) ? last1 : last0) ? sc[nt][c] * scale_log2 : -CUDART_INF_F;
      }
    } else {
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int key = gq + ((c >> 1) << 3);
        sc[nt][c] = key < valid ? sc[nt][c] * scale_log2 : -CUDART_INF_F;
      }
    }
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float mx = fmaxf(sc[nt][j], sc[nt][j + 2]);
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(st.m_run[nt][j], mx);
      const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
      alpha[nt][j] = ptx::ex2(st.m_run[nt][j] - m_use);
      st.m_run[nt][j] = m_new;
      const float p0 = ptx::ex2(sc[nt][j] - m_use);
      const float p1 = ptx::ex2(sc[nt][j + 2] - m_use);
      st.l_run[nt][j] = st.l_run[nt][j] * alpha[nt][j] + (p0 + p1);
      sc[nt][j] = p0;
      sc[nt][j + 2] = p1;
    }
  }
  // ---- rescale O^T (rows d, columns = query rows 2*tq4, 2*tq4+1); skipped when no
  //      running max of the warp moved (alpha = 1 everywhere), the common case once the
  //      first tiles have been seen (G*T_q = 32: 94.5 -> 92.9 us; no change at G*T_q = 4)
  bool moved = false;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) moved |= (alpha[nt][0] != 1.f) | (alpha[nt][1] != 1.f);
  if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
    for (int i = 0; i < KD; ++i)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        st.acc[i][nt][0] *= alpha[nt][0];
        st.acc[i][nt][1] *= alpha[nt][1];
        st.acc[i][nt][2] *= alpha[nt][0];
        st.acc[i][nt][3] *= alpha[nt][1];
      }
  }
  // ---- P^T as the B operand (keys x query rows): transpose 8x8 f16 blocks in registers
  uint32_t pf[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    pf[nt][0] = ptx::movmatrix_trans(Elem<BF16>::pack(sc[nt][0], sc[nt][1]));
    pf[nt][1] = ptx::movmatrix_trans(Elem<BF16>::pack(sc[nt][2], sc[nt][3]));
  }
  // ---- O^T += V^T P^T
#pragma unroll
  for (int i = 0; i < KD; ++i) {
    uint32_t af[4];
    if constexpr (VLLM) {
      // V^T is stored: rows d 16i .. 16i+15, 8 keys per ldmatrix row
      ptx::ldmatrix_x4(af, smem_clamp(vvb + vllm_v_offset(i * 16 + v_dr, v_kb, rb), 16, ring.lo, ring.hi,
                                      ring.status));
    } else {
      ptx::ldmatrix_x4_trans(af, smem_clamp(chunk_addr(vbase, v_off, v_row, i * 2 + v_c0, plane), 16, ring.lo,
                                            ring.hi, ring.status));
    }
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) Elem<BF16>::mma(st.acc[i][nt], af, pf[nt]);
  }
}

// Two 16-key slices of one stage at once (row layout): the warp's slices ks[0] and ks[1] of a
// stage of two 64-key tiles (d_head 64), with the same arithmetic as consume_tile on both -- the
// two slices' S products in flight together, one running-max update, rescale and l update for the
// 32 keys, then both P.V products -- so that the two slices' dependent chains overlap instead of
// running back to back.  Slice 1 holds keys (valid[1] > 0) only when slice 0 is whole.
template <int D, int NT, int BOXP, bool CAUSAL = false, bool BF16 = false>
__device__ __forceinline__ void consume_tile2(WarpState<D, NT>& st, uint32_t kbase, uint32_t vbase,
                                              const int (&valid)[2], const int (&key0)[2], const int (&ks)[2],
                                              int lane, float scale_log2, int rb, const Win& ring) {
  constexpr int KD = WarpState<D, NT>::KD;
  const int gq = lane >> 2;
  const int k_c0 = lane >> 4;
  const int v_c0 = (lane >> 3) & 1;
  const int plane = rb * 128;
  int k_row[2], v_row[2], k_off[2], v_off[2];
#pragma unroll
  for (int u = 0; u < 2; ++u) {
    k_row[u] = ks[u] * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
    v_row[u] = ks[u] * 16 + (lane & 7) + ((lane >> 4) & 1) * 8;
    k_off[u] = row_offset<BOXP>(k_row[u], rb);
    v_off[u] = row_offset<BOXP>(v_row[u], rb);
  }

  // ---- S^T = K Q^T for both slices: 2 x 16 keys x 8*NT query rows, fp32
  float sc[2][NT][4];
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) sc[u][nt][0] = sc[u][nt][1] = sc[u][nt][2] = sc[u][nt][3] = 0.f;
#pragma unroll
  for (int kk = 0; kk < KD; ++kk) {
    uint32_t af[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
      ptx::ldmatrix_x4(af[u], smem_clamp(chunk_addr(kbase, k_off[u], k_row[u], kk * 2 + k_c0, plane), 16, ring.lo,
                                         ring.hi, ring.status));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      Elem<BF16>::mma(sc[0][nt], af[0], st.qf[nt][kk]);
      Elem<BF16>::mma(sc[1][nt], af[1], st.qf[nt][kk]);
    }
  }
  // ---- scale (log2 domain) and mask each slice; sc[u][nt][c]: key gq (c<2) or gq+8 of slice u,
  //      query row 2*tq4 + (c&1) of n-tile nt
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      if constexpr (CAUSAL) {
        const int last0 = min(valid[u] - 1, st.lim[nt][0] - key0[u]);
        const int last1 = min(valid[u] - 1, st.lim[nt][1] - key0[u]);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int key = gq + ((c >> 1) << 3);
          sc[u][nt][c] = key <= ((c & 1) ? last1 : last0) ? sc[u][nt][c] * scale_log2 : -CUDART_INF_F;
        }
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int key = gq + ((c >> 1) << 3);
          sc[u][nt][c] = key < valid[u] ? sc[u][nt][c] * scale_log2 : -CUDART_INF_F;
        }
      }
    }
  // ---- online softmax over the 32 keys
  float alpha[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float mx = fmaxf(fmaxf(sc[0][nt][j], sc[0][nt][j + 2]), fmaxf(sc[1][nt][j], sc[1][nt][j + 2]));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(st.m_run[nt][j], mx);
      const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
      alpha[nt][j] = ptx::ex2(st.m_run[nt][j] - m_use);
      st.m_run[nt][j] = m_new;
      const float p00 = ptx::ex2(sc[0][nt][j] - m_use), p01 = ptx::ex2(sc[0][nt][j + 2] - m_use);
      const float p10 = ptx::ex2(sc[1][nt][j] - m_use), p11 = ptx::ex2(sc[1][nt][j + 2] - m_use);
      st.l_run[nt][j] = st.l_run[nt][j] * alpha[nt][j] + ((p00 + p01) + (p10 + p11));
      sc[0][nt][j] = p00;
      sc[0][nt][j + 2] = p01;
      sc[1][nt][j] = p10;
      sc[1][nt][j + 2] = p11;
    }
  // ---- rescale O^T when a running max of the warp moved (as consume_tile)
  bool moved = false;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) moved |= (alpha[nt][0] != 1.f) | (alpha[nt][1] != 1.f);
  if (__any_sync(0xffffffffu, moved)) {
#pragma unroll
    for (int i = 0; i < KD; ++i)
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        st.acc[i][nt][0] *= alpha[nt][0];
        st.acc[i][nt][1] *= alpha[nt][1];
        st.acc[i][nt][2] *= alpha[nt][0];
        st.acc[i][nt][3] *= alpha[nt][1];
      }
  }
  // ---- P^T of both slices as B operands
  uint32_t pf[2][NT][2];
#pragma unroll
  for (int u = 0; u < 2; ++u)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      pf[u][nt][0] = ptx::movmatrix_trans(Elem<BF16>::pack(sc[u][nt][0], sc[u][nt][1]));
      pf[u][nt][1] = ptx::movmatrix_trans(Elem<BF16>::pack(sc[u][nt][2], sc[u][nt][3]));
    }
  // ---- O^T += V^T P^T, slice 0 then slice 1 into each accumulator
#pragma unroll
  for (int i = 0; i < KD; ++i) {
    uint32_t af[2][4];
#pragma unroll
    for (int u = 0; u < 2; ++u)
      ptx::ldmatrix_x4_trans(af[u], smem_clamp(chunk_addr(vbase, v_off[u], v_row[u], i * 2 + v_c0, plane), 16,
                                               ring.lo, ring.hi, ring.status));
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      Elem<BF16>::mma(st.acc[i][nt], af[0], pf[0][nt]);
      Elem<BF16>::mma(st.acc[i][nt], af[1], pf[1][nt]);
    }
  }
}

// =====================================================================================
// end of a slice: merge the key-slice warps, emit, merge the unit's slices
// =====================================================================================

// Reduce l over the lanes that share a query row and write this warp's (O, m, l)
// into its block of the shared-memory scratch.
template <int D, int NT, int WN, int STAGES>
__device__ __forceinline__ void stash_warp(WarpState<D, NT>& st, float* scratch, int warp, int lane,
                                           uint32_t* status) {
  using C = Cfg<D, NT, WN, STAGES>;
  // every index below stays inside this warp's block of the scratch: check the block once
  if (!idx_ok((int64_t)(warp + 1) * C::WSCRATCH - 1, (int64_t)C::CONSUMERS * C::WSCRATCH, status)) return;
  const int gq = lane >> 2, tq4 = lane & 3;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float l = st.l_run[nt][j];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      st.l_run[nt][j] = l;
    }
  float* wsp = scratch + warp * C::WSCRATCH;
  float* wm = wsp + C::WROWS * C::OSTRIDE;
  float* wl = wm + C::WROWS;
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int r0 = nt * 8 + 2 * tq4;
#pragma unroll
    for (int i = 0; i < WarpState<D, NT>::KD; ++i) {
      wsp[r0 * C::OSTRIDE + i * 16 + gq] = st.acc[i][nt][0];
      wsp[(r0 + 1) * C::OSTRIDE + i * 16 + gq] = st.acc[i][nt][1];
      wsp[r0 * C::OSTRIDE + i * 16 + gq + 8] = st.acc[i][nt][2];
      wsp[(r0 + 1) * C::OSTRIDE + i * 16 + gq + 8] = st.acc[i][nt][3];
    }
    if (gq == 0) {
      wm[r0] = st.m_run[nt][0];
      wm[r0 + 1] = st.m_run[nt][1];
      wl[r0] = st.l_run[nt][0];
      wl[r0 + 1] = st.l_run[nt][1];
    }
  }
}

// Combine the key-slice warps of every query row of the item's HG KV heads (g0 ..
// g0+HG-1) and emit: the final f16 output (single slice), the caller's partial (single
// slice, partial mode) or this slice's fp32 partial in the workspace.  With HG heads a
// head has kWK/HG key-slice warps (hh*KS .. hh*KS+KS-1); with one head, warp col*kWK+k
// holds key slice k of query column col.
// The KS key-slice warps w0 .. w0+KS-1 of one query row (row lr of each warp's block) folded
// into one (M, L, O[d]) -- M in the log2 domain of the scaled logits.
template <int D, int NT, int WN, int STAGES, int KS>
__device__ __forceinline__ void combine_warps(const float* scratch, int w0, int lr, int d, float& M, float& L,
                                              float& O, uint32_t* status) {
  using C = Cfg<D, NT, WN, STAGES>;
  float mk[KS];
  M = -CUDART_INF_F;
  L = 0.f;
  O = 0.f;
  // the KS warps' blocks, and row lr / column d inside a block
  if (!idx_ok((int64_t)(w0 + KS) * C::WSCRATCH - 1, (int64_t)C::CONSUMERS * C::WSCRATCH, status) ||
      !idx_ok(lr, C::WROWS, status) || !idx_ok(d, D, status))
    return;
#pragma unroll
  for (int k = 0; k < KS; ++k) {
    const float* wsp = scratch + (w0 + k) * C::WSCRATCH;
    mk[k] = wsp[C::WROWS * C::OSTRIDE + lr];
    M = fmaxf(M, mk[k]);
  }
  L = 0.f;
  O = 0.f;
  if (M != -CUDART_INF_F) {
#pragma unroll
    for (int k = 0; k < KS; ++k) {
      const float* wsp = scratch + (w0 + k) * C::WSCRATCH;
      const float w = ptx::ex2(mk[k] - M);
      L += w * wsp[C::WROWS * C::OSTRIDE + C::WROWS + lr];
      O += w * wsp[lr * C::OSTRIDE + d];
    }
  }
}

template <int D, int NT, int WN, int STAGES, int HG = 1, bool BF16 = false>
__device__ __forceinline__ void emit_slice(const DecodeArgs& a, const float* scratch, int b, int g0, int slice,
                                           bool single, int tid, int nthreads) {
  using C = Cfg<D, NT, WN, STAGES>;
  constexpr int KS = kWK / HG;
  const int per_head = a.rows * D;
  for (int idx = tid; idx < HG * per_head; idx += nthreads) {
    const int hh = idx / per_head;
    const int rem = idx - hh * per_head;
    const int r = rem / D, d = rem - r * D;
    const int col = r / C::WROWS, lr = r - col * C::WROWS;
    const int w0 = HG > 1 ? hh * KS : col * kWK;
    const int g = g0 + hh;
    float M, L, O;
    combine_warps<D, NT, WN, STAGES, KS>(scratch, w0, lr, d, M, L, O, a.status);
    const int64_t orow = out_row(a, b, g, r);
    if (!idx_ok(orow, a.R, a.status)) continue;
    if (single) {
      if (a.o != nullptr) {
        Elem<BF16>::store(a.o, orow * D + d, L > 0.f ? O / L : 0.f);
      } else {
        if (d == 0) {
          a.m_out[orow] = M * kLn2;
          a.l_out[orow] = L;
        }
        a.o_part_out[orow * D + d] = O;
      }
    } else {
      const int64_t prow = (int64_t)slice * a.R + orow;
      if (!idx_ok(slice, a.n_splits, a.status)) continue;
      if (d == 0) {
        a.ws_m[prow] = M * kLn2;
        a.ws_l[prow] = L;
      }
      a.ws_o[prow * D + d] = O;
    }
  }
}

// The same for one warp (the paged kernel's epilogue warp): a row per step, each lane folding and
// writing D/32 consecutive columns, so that the output row's index arithmetic runs once per row
// and the stores are 8- or 16-byte vectors.  (One element per lane per step took this warp ~15 us
// per 512-key item of 4 KV heads on GB300 -- most of the time the item streams.)
template <int D, int NT, int WN, int STAGES, int HG = 1, bool BF16 = false>
__device__ __forceinline__ void emit_slice_warp(const DecodeArgs& a, const float* scratch, int b, int g0, int slice,
                                                bool single, int lane) {
  using C = Cfg<D, NT, WN, STAGES>;
  constexpr int KS = kWK / HG;
  constexpr int PER = D / 32;                          // 4 columns (d 128) or 2 (d 64) per lane
  if (!single && !idx_ok(slice, a.n_splits, a.status)) return;
  for (int hh = 0; hh < HG; ++hh) {
    for (int r = 0; r < a.rows; ++r) {
      const int col = r / C::WROWS, lr = r - col * C::WROWS;
      const int w0 = HG > 1 ? hh * KS : col * kWK;
      if (!idx_ok((int64_t)(w0 + KS) * C::WSCRATCH - 1, (int64_t)C::CONSUMERS * C::WSCRATCH, a.status)) return;
      float mk[KS];
      float M = -CUDART_INF_F;
#pragma unroll
      for (int k = 0; k < KS; ++k) {
        mk[k] = scratch[(w0 + k) * C::WSCRATCH + C::WROWS * C::OSTRIDE + lr];
        M = fmaxf(M, mk[k]);
      }
      float L = 0.f, o[PER];
#pragma unroll
      for (int i = 0; i < PER; ++i) o[i] = 0.f;
      if (M != -CUDART_INF_F) {
#pragma unroll
        for (int k = 0; k < KS; ++k) {
          const float* wsp = scratch + (w0 + k) * C::WSCRATCH;
          const float w = ptx::ex2(mk[k] - M);
          L += w * wsp[C::WROWS * C::OSTRIDE + C::WROWS + lr];
#pragma unroll
          for (int i = 0; i < PER; ++i) o[i] += w * wsp[lr * C::OSTRIDE + lane * PER + i];
        }
      }
      const int64_t orow = out_row(a, b, g0 + hh, r);
      if (!idx_ok(orow, a.R, a.status)) continue;
      if (single) {
        // a one-partition sequence: the final output
        const float inv = L > 0.f ? 1.f / L : 0.f;
        uint32_t pk[PER / 2];
#pragma unroll
        for (int i = 0; i < PER / 2; ++i) pk[i] = Elem<BF16>::pack(o[2 * i] * inv, o[2 * i + 1] * inv);
        __half* dst = a.o + orow * D + lane * PER;
        if constexpr (PER == 4) {
          *reinterpret_cast<uint2*>(dst) = make_uint2(pk[0], pk[1]);
        } else {
          *reinterpret_cast<uint32_t*>(dst) = pk[0];
        }
      } else {
        const int64_t prow = (int64_t)slice * a.R + orow;
        if (lane == 0) {
          a.ws_m[prow] = M * kLn2;
          a.ws_l[prow] = L;
        }
        float* dst = a.ws_o + prow * D + lane * PER;
        if constexpr (PER == 4) {
          *reinterpret_cast<float4*>(dst) = make_float4(o[0], o[1], o[2], o[3]);
        } else {
          *reinterpret_cast<float2*>(dst) = make_float2(o[0], o[1]);
        }
      }
    }
  }
}

// After this slice's partial is written: take an arrival ticket for the unit; true
// on the CTA that arrives last (all other slices of the unit are then in memory).
template <int CTHREADS>
__device__ __forceinline__ bool last_to_arrive(const DecodeArgs& a, int unit, int n_slices, volatile int* flags) {
  __threadfence();
  ptx::named_bar_sync(1, CTHREADS);
  if (threadIdx.x == 0) {
    flags[1] = 0;
    if (idx_ok(unit, (int64_t)a.B * a.h_kv, a.status)) {
      const unsigned prev = atomicAdd(a.counters + unit, 1u);
      flags[1] = (prev == (unsigned)(n_slices - 1)) ? 1 : 0;
    }
  }
  ptx::named_bar_sync(1, CTHREADS);
  const bool last = flags[1] != 0;
  if (last) __threadfence();
  return last;
}

// Fold the n partials of unit (b, g) (page: _merge_running applied left to right) for the
// items item0 + threadIdx.x + i * NTH (i < IPT; an item is 4 consecutive d of one query
// row) and write the output (O / l) or the merged partial.  Partials are read in chunks
// whose loads are all issued before the folds.
template <int D, int NTH, int IPT, bool BF16>
__device__ __forceinline__ void merge_pass(const DecodeArgs& a, int b, int g, int item0, int n) {
  constexpr int DQ = D / 4;
  const int n_items = a.rows * DQ;
  float M[IPT], L[IPT];
  float4 O[IPT];
  int64_t orow_i[IPT];
  int c4_i[IPT];
  bool ok_i[IPT];
#pragma unroll
  for (int i = 0; i < IPT; ++i) {
    const int item = item0 + threadIdx.x + i * NTH;
    const int r = item < n_items ? item / DQ : 0;
    c4_i[i] = item < n_items ? item - r * DQ : 0;
    orow_i[i] = out_row(a, b, g, r);
    ok_i[i] = idx_ok(orow_i[i], a.R, a.status);
    if (!ok_i[i]) orow_i[i] = 0;   // read in range, nothing written for it below
    M[i] = -CUDART_INF_F;
    L[i] = 0.f;
    O[i] = make_float4(0.f, 0.f, 0.f, 0.f);
  }
  // chunks of UNR partials: all UNR x IPT loads are issued before any is used, about 16
  // float4 loads in flight per thread
  constexpr int UNR = IPT >= 4 ? 4 : 16 / IPT;
  if (n > 0 && !idx_ok(n - 1, a.n_splits, a.status)) n = 0;   // only this call's splits' partials are read
  for (int s0 = 0; s0 < n; s0 += UNR) {
    float ms[UNR][IPT], ls[UNR][IPT];
    float4 os[UNR][IPT];
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
      const bool have = s0 + u < n;
#pragma unroll
      for (int i = 0; i < IPT; ++i) {
        const int64_t prow = (int64_t)(have ? s0 + u : 0) * a.R + orow_i[i];
        ms[u][i] = have ? __ldcg(a.ws_m + prow) * kLog2e : -CUDART_INF_F;
        ls[u][i] = have ? __ldcg(a.ws_l + prow) : 0.f;
        os[u][i] = have ? __ldcg(reinterpret_cast<const float4*>(a.ws_o + prow * D) + c4_i[i])
                        : make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
#pragma unroll
    for (int u = 0; u < UNR; ++u) {
#pragma unroll
      for (int i = 0; i < IPT; ++i) {
        const float m_new = fmaxf(M[i], ms[u][i]);
        const float ref = m_new == -CUDART_INF_F ? 0.f : m_new;   // both sides empty so far
        const float so = ptx::ex2(M[i] - ref), sn = ptx::ex2(ms[u][i] - ref);
        L[i] = L[i] * so + ls[u][i] * sn;
        O[i].x = O[i].x * so + os[u][i].x * sn;
        O[i].y = O[i].y * so + os[u][i].y * sn;
        O[i].z = O[i].z * so + os[u][i].z * sn;
        O[i].w = O[i].w * so + os[u][i].w * sn;
        M[i] = m_new;
      }
    }
  }
#pragma unroll
  for (int i = 0; i < IPT; ++i) {
    if (item0 + threadIdx.x + i * NTH >= n_items) continue;
    if (!ok_i[i]) continue;
    const int64_t orow = orow_i[i];
    if (a.o != nullptr) {
      const float inv = L[i] > 0.f ? 1.f / L[i] : 0.f;
      Elem<BF16>::store2(a.o, orow * D + c4_i[i] * 4, O[i].x * inv, O[i].y * inv);
      Elem<BF16>::store2(a.o, orow * D + c4_i[i] * 4 + 2, O[i].z * inv, O[i].w * inv);
    } else {
      if (c4_i[i] == 0) {
        a.m_out[orow] = M[i] * kLn2;
        a.l_out[orow] = L[i];
      }
      reinterpret_cast<float4*>(a.o_part_out + orow * D)[c4_i[i]] = O[i];
    }
  }
}

// The whole unit in one pass (each consumer thread IPT items); resets the unit's counter.
template <int D, int NT, int WN, int STAGES, bool BF16 = false>
__device__ __forceinline__ void merge_unit(const DecodeArgs& a, int b, int g, int unit, int n) {
  using C = Cfg<D, NT, WN, STAGES>;
  constexpr int IPT = (C::WROWS * WN * (D / 4) + C::CTHREADS - 1) / C::CTHREADS;
  merge_pass<D, C::CTHREADS, IPT, BF16>(a, b, g, 0, n);
  if (threadIdx.x == 0 && idx_ok(unit, (int64_t)a.B * a.h_kv, a.status)) atomicExch(a.counters + unit, 0u);
}

// =====================================================================================
// merge inside a thread-block cluster: the splits of one unit are the CTAs of one cluster
// =====================================================================================
// Largest cluster of the split kernel's cluster variant: 16 CTAs (beyond the portable 8, allowed
// per kernel with cudaFuncAttributeNonPortableClusterSizeAllowed).
constexpr int kMaxClusterSplits = 16;
static_assert(kMaxClusterSplits <= 32, "the cluster fold checks the CTAs' flags one per lane of a warp");

// The receiving area of a CTA of the cluster variant, in shared memory of its own (apart from the
// ring, which siblings may still be filling when they push): the unit's items -- (row, 4 columns)
// pairs -- are dealt out to the n CTAs in contiguous runs of at most ipo = ceil(items / n), and
// every CTA pushes its partial of each item to the item's owner: float4 O [n][ipo] and
// float2 (m, l) [n][ipo] (m in the log2 domain), source-major, plus the sources' completion flags.
template <int RMAX, int D>
struct ClusterRecv {
  static constexpr int ITEMS = RMAX * (D / 4);
  static constexpr int SLOTS = ITEMS + kMaxClusterSplits;   // n * ipo <= items + n - 1
  static constexpr int O = 0;
  static constexpr int ML = SLOTS * 16;
  static constexpr int VALID = ML + SLOTS * 8;
  static constexpr int BYTES = VALID + kMaxClusterSplits * 4;
};

// Items [first, end) of the unit's n_items that CTA `rank` of n owns, and the owner of an item:
// ceil(rank * n_items / n) <= item < ceil((rank + 1) * n_items / n)  <=>  owner = floor(item * n / n_items).
// 32-bit arithmetic: n_items <= 64 rows x 32 column groups, n <= kMaxClusterSplits (the 64-bit
// divisions took a quarter of a microsecond of the fold).
__device__ __forceinline__ int cluster_first_item(int rank, int n, int n_items) {
  return (rank * n_items + n - 1) / n;
}

// This CTA's partial of every item of the unit, its key-slice warps folded, pushed into the
// owners' receiving areas through distributed shared memory (the stores are complete, for the
// owners, once the cluster barrier that follows has been passed).  `recv`: the receiving area's
// shared-memory address, the same offset in every CTA.
template <int D, int NT, int WN, int STAGES>
__device__ __forceinline__ void push_cta_partial(const DecodeArgs& a, const float* scratch, uint32_t recv, int n,
                                                 int rank, int tid, int nthreads) {
  using C = Cfg<D, NT, WN, STAGES>;
  using RV = ClusterRecv<C::WROWS * WN, D>;
  constexpr int DQ = D / 4;
  const int n_items = a.rows * DQ;
  const int ipo = (n_items + n - 1) / n;
  for (int idx = tid; idx < n_items; idx += nthreads) {
    const int r = idx / DQ, c4 = idx - r * DQ;
    const int col = r / C::WROWS, lr = r - col * C::WROWS;
    const int w0 = col * kWK;
    if (!idx_ok((int64_t)(w0 + kWK) * C::WSCRATCH - 1, (int64_t)C::CONSUMERS * C::WSCRATCH, a.status) ||
        !idx_ok(lr, C::WROWS, a.status))
      continue;
    // the kWK key-slice warps of row r, columns 4 c4 .. 4 c4 + 3
    float mk[kWK];
    float M = -CUDART_INF_F;
#pragma unroll
    for (int k = 0; k < kWK; ++k) {
      mk[k] = scratch[(w0 + k) * C::WSCRATCH + C::WROWS * C::OSTRIDE + lr];
      M = fmaxf(M, mk[k]);
    }
    float L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int k = 0; k < kWK; ++k) {
        const float* wsp = scratch + (w0 + k) * C::WSCRATCH;
        const float w = ptx::ex2(mk[k] - M);
        L += w * wsp[C::WROWS * C::OSTRIDE + C::WROWS + lr];
        const float4 o = *reinterpret_cast<const float4*>(wsp + lr * C::OSTRIDE + c4 * 4);
        O.x += w * o.x;
        O.y += w * o.y;
        O.z += w * o.z;
        O.w += w * o.w;
      }
    }
    const int owner = idx * n / n_items;
    const int j = idx - cluster_first_item(owner, n, n_items);
    const int slot = rank * ipo + j;
    if (!idx_ok(slot, RV::SLOTS, a.status) || !idx_ok(owner, n, a.status)) continue;
    const uint32_t dst = ptx::mapa(recv, (uint32_t)owner);
    ptx::st_cluster_v4(dst + RV::O + slot * 16, O);
    ptx::st_cluster_v2(dst + RV::ML + slot * 8, M, L);
  }
}

// One online-softmax merge step of two partials (M in the log2 domain): the page's
// _merge_running, both sides rescaled to the larger max; empty sides (M = -inf) contribute nothing.
__device__ __forceinline__ void merge_into(float& M, float& L, float4& O, float m2, float l2, const float4& o2) {
  const float m_new = fmaxf(M, m2);
  const float ref = m_new == -CUDART_INF_F ? 0.f : m_new;   // both sides empty so far
  const float so = ptx::ex2(M - ref), sn = ptx::ex2(m2 - ref);
  L = L * so + l2 * sn;
  O.x = O.x * so + o2.x * sn;
  O.y = O.y * so + o2.y * sn;
  O.z = O.z * so + o2.z * sn;
  O.w = O.w * so + o2.w * sn;
  M = m_new;
}

// After the cluster barrier: fold, for this CTA's items, the n sources' partials it received (the
// page's _merge_running, then O / l) from its own shared memory, and write the output (or the
// merged partial).  An item's sources are spread over a group of `lpi` lanes (a power of two, up to
// 16, as many as the CTA's threads allow): lane k of the group folds sources k, k + lpi, ... in
// order, then the group combines its lanes in a fixed butterfly of shuffles -- a fixed order, so
// results are reproducible; one thread walking all 16 sources took ~1 us for the tiny workload.
// (The closed form -- the group's max first, one exponential per source, then the group's sums --
// measured slower on GB300: tiny workload 4.39 -> 4.62 us per L2-resident step, two serial
// butterflies against one.)
// Nothing is written unless every CTA completed its slice (a wait that gave up leaves the output
// alone).
template <int RMAX, int D, int NTH, bool BF16>
__device__ __forceinline__ void fold_received(const DecodeArgs& a, int b, int g, const uint8_t* recv, int n,
                                              int rank) {
  using RV = ClusterRecv<RMAX, D>;
  constexpr int DQ = D / 4;
  const int lane = threadIdx.x & 31;
  const int flag = lane < n ? reinterpret_cast<const volatile int*>(recv + RV::VALID)[lane] : 1;
  if (!__all_sync(0xffffffffu, flag != 0)) return;
  const int n_items = a.rows * DQ;
  const int ipo = (n_items + n - 1) / n;
  const int lo = cluster_first_item(rank, n, n_items), hi = cluster_first_item(rank + 1, n, n_items);
  int lg = 0;   // lanes per item: 1 << lg
  while (lg < 4 && (1 << lg) < n && (hi - lo) << (lg + 1) <= NTH) ++lg;
  const int lpi = 1 << lg;
  const int sub = (int)threadIdx.x & (lpi - 1);
  const float4* ro = reinterpret_cast<const float4*>(recv + RV::O);
  const float2* rml = reinterpret_cast<const float2*>(recv + RV::ML);
  // every thread runs the same number of rounds, so that whole warps meet at the shuffles
  for (int base = lo; base < hi; base += NTH >> lg) {
    const int item = base + ((int)threadIdx.x >> lg);
    const int j = item - lo;
    const bool mine = item < hi && idx_ok((int64_t)(n - 1) * ipo + j, RV::SLOTS, a.status);
    float M = -CUDART_INF_F, L = 0.f;
    float4 O = make_float4(0.f, 0.f, 0.f, 0.f);
    if (mine)
      for (int s = sub; s < n; s += lpi) {
        const float2 ml = rml[s * ipo + j];
        merge_into(M, L, O, ml.x, ml.y, ro[s * ipo + j]);
      }
    for (int off = lpi >> 1; off > 0; off >>= 1) {   // the group's butterfly
      const float m2 = __shfl_xor_sync(0xffffffffu, M, off), l2 = __shfl_xor_sync(0xffffffffu, L, off);
      float4 o2;
      o2.x = __shfl_xor_sync(0xffffffffu, O.x, off);
      o2.y = __shfl_xor_sync(0xffffffffu, O.y, off);
      o2.z = __shfl_xor_sync(0xffffffffu, O.z, off);
      o2.w = __shfl_xor_sync(0xffffffffu, O.w, off);
      // both lanes of a pair fold (lower lane's partial, upper lane's) in that order: the same
      // result on both, selected rather than branched on so the pair does not diverge
      const bool upper = (threadIdx.x & off) != 0;
      float M1 = upper ? m2 : M, L1 = upper ? l2 : L;
      float4 O1 = upper ? o2 : O;
      const float M2 = upper ? M : m2, L2 = upper ? L : l2;
      const float4 O2 = upper ? O : o2;
      merge_into(M1, L1, O1, M2, L2, O2);
      M = M1;
      L = L1;
      O = O1;
    }
    if (!mine || sub != 0) continue;
    const int r = item / DQ, c4 = item - r * DQ;
    if (!idx_ok(r, RMAX, a.status) || !idx_ok(out_row(a, b, g, r), a.R, a.status)) continue;
    const int64_t orow = out_row(a, b, g, r);
    if (a.o != nullptr) {
      const float inv = L > 0.f ? 1.f / L : 0.f;
      Elem<BF16>::store2(a.o, orow * D + c4 * 4, O.x * inv, O.y * inv);
      Elem<BF16>::store2(a.o, orow * D + c4 * 4 + 2, O.z * inv, O.w * inv);
    } else {
      if (c4 == 0) {
        a.m_out[orow] = M * kLn2;
        a.l_out[orow] = L;
      }
      reinterpret_cast<float4*>(a.o_part_out + orow * D)[c4] = O;
    }
  }
}

// =====================================================================================
// contiguous K/V: one CTA per (KV head, split, sequence)
// =====================================================================================
// 64-key tiles per pipeline stage of the split kernel: two at d_head 64, so that a stage (one
// 128-row TMA box of K and one of V, 32 KB) amortises the per-stage waits and barriers over as
// many bytes as a 64-key stage at d_head 128 (measured on GB300 at 2^18 keys, 8 KV heads,
// d_head 64: 4 query rows 111.3 -> 94.9 us, 8 rows 113.3 -> 96.9 us)
__host__ __device__ constexpr int split_sub(int D) { return D == 64 ? 2 : 1; }

// CLUSTER: launched with cluster dimensions (1, n_splits, 1) -- the splits of a unit are the CTAs
// of one cluster, which exchange their partials through distributed shared memory in place of the
// workspace and the arrival ticket (every thread of every CTA takes part in both phases of the
// cluster barrier: one before the first remote store, one after the last).
template <int D, int NT, int WN, int STAGES, int SUB, bool CAUSAL, bool BF16, bool CLUSTER = false>
__global__ void __launch_bounds__(Cfg<D, NT, WN, STAGES * SUB>::THREADS)
gqa_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const DecodeArgs a) {
  // sizes of a ring of STAGES stages of SUB 64-key tiles (the Cfg of STAGES * SUB single tiles)
  using C = Cfg<D, NT, WN, STAGES * SUB>;
  constexpr int KVB = SUB * C::KV_BYTES;     // K (or V) bytes of one stage
  constexpr int STB = 2 * KVB;               // one stage
  constexpr int SROWS = SUB * kTile;         // keys (TMA box rows) per stage
  // CLUSTER: the receiving area, after the barriers and flags (split_smem_bytes counts it)
  constexpr int RECV_OFF = C::DATA_BYTES + ((C::CTRL_BYTES + 15) & ~15);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::DATA_BYTES);
  uint64_t* empty = full + STAGES;
  // [0] abort, [1] last-CTA, [2] CLUSTER: this CTA's partial is complete
  volatile int* flags = reinterpret_cast<volatile int*>(empty + STAGES);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g_kv = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
  const int unit = b * a.h_kv + g_kv;
  const Win ring{ptx::smem_u32(smem), ptx::smem_u32(smem) + (uint32_t)C::PIPE_BYTES, a.status};

  // ---- this CTA's key range [key_begin, key_end)
  const int64_t tiles_total = (a.s_len + kTile - 1) / kTile;
  const int64_t t0 = tiles_total * split / a.n_splits;
  const int64_t t1 = tiles_total * (split + 1) / a.n_splits;
  const int64_t key_begin = a.s_begin + t0 * kTile;
  const int64_t key_end = min(a.s_begin + t1 * kTile, a.s_begin + a.s_len);
  const int n_tiles = (int)((t1 - t0 + SUB - 1) / SUB);   // stages
  const int64_t y_base = (int64_t)b * a.S_kv;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(full + s), 1);
      ptx::mbar_init(ptx::smem_u32(empty + s), C::CONSUMERS);
    }
    flags[0] = 0;
    flags[1] = 0;
    flags[2] = 0;
    ptx::fence_mbar_init();
  }
  if (warp == C::CONSUMERS && lane == 0) {
    ptx::prefetch_tensormap(&tmK);
    ptx::prefetch_tensormap(&tmV);
  }
  __syncthreads();
  // CLUSTER: first phase of the cluster barrier, waited for before the first access to another
  // CTA's shared memory (which must be running by then); every CTA arrives here, long before
  if constexpr (CLUSTER) ptx::cluster_arrive_relaxed();
  // the first ring's worth of K and V boxes into L2 while the previous kernel in the stream may
  // still run (a hint: the loads below, after the dependency wait, read whatever it wrote).  Only
  // for sweeps longer than the ring: measured on GB300 (us per step, without / with): ragged
  // 81.33 / 80.50 and verify16 167.9 / 166.5 (tcgen05 kernel), long 569.07 / 567.37, llama8b
  // 147.9 / 147.6; the tiny workload's L2-resident steps, whose splits fit in the ring, lost 0.12 us
  if (warp == C::CONSUMERS && lane == 0 && n_tiles > STAGES) {
    for (int it = 0; it < n_tiles && it < STAGES; ++it) {
      const int64_t y = y_base + key_begin + (int64_t)it * SROWS;
      if (y < (int64_t)a.B * a.S_kv && g_kv < a.h_kv) {
        ptx::tma_prefetch_3d(&tmK, 0, (int)y, g_kv * C::HALVES);
        ptx::tma_prefetch_3d(&tmV, 0, (int)y, g_kv * C::HALVES);
      }
    }
  }
  // launched as a programmatic dependent: the set-up above may overlap the previous kernel in the
  // stream; nothing in global memory is read or written before that kernel has completed
  ptx::grid_dependency_wait();

  // ---------------------------------------------------------------- producer warp
  if (warp == C::CONSUMERS) {
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_first();
      const int stall_tile = (a.stall_cta >= 0 &&
                              a.stall_cta == (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z)))
                                 ? 1 : -1;
      int issued = 0;
      bool gave_up = false;
      for (int it = 0; it < n_tiles; ++it) {
        const int s = it % STAGES;
        const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
        if (it >= STAGES && !ptx::mbar_wait_bounded(ptx::smem_u32(empty + s), ph ^ 1u, a.timeout_ns, flags)) {
          raise_timeout(a, flags);
          gave_up = true;
          break;
        }
        issued = it + 1;
        if (it == stall_tile) continue;  // test hook: this tile is never loaded
        const uint32_t kdst = ptx::smem_u32(smem + s * STB);
        const uint32_t vdst = kdst + KVB;
        const uint32_t fb = ptx::smem_u32(full + s);
        const int64_t y = y_base + key_begin + (int64_t)it * SROWS;
        // the box starts inside K / V's rows and heads and lands inside the ring (else the stage
        // completes without data: the check has recorded it)
        if (idx_ok(y, (int64_t)a.B * a.S_kv, a.status) && idx_ok(g_kv, a.h_kv, a.status) &&
            smem_ok(kdst, STB, ring.lo, ring.hi, a.status)) {
          ptx::mbar_arrive_expect_tx(fb, STB);
          ptx::tma_load_3d(kdst, &tmK, fb, 0, (int)y, g_kv * C::HALVES, pol);
          ptx::tma_load_3d(vdst, &tmV, fb, 0, (int)y, g_kv * C::HALVES, pol);
        } else {
          ptx::mbar_arrive(fb);
        }
      }
      if (gave_up || stall_tile >= 0) {
        // wait (bounded) for copies still in flight before the CTA can exit
        for (int it = max(0, issued - STAGES); it < issued; ++it) {
          if (it == stall_tile) continue;
          ptx::mbar_wait_bounded(ptx::smem_u32(full + (it % STAGES)), (uint32_t)(it / STAGES) & 1u,
                                 a.timeout_ns, nullptr);
        }
      }
    }
    if constexpr (CLUSTER) {   // the producer's threads take part in both cluster barrier phases too
      __syncwarp();
      ptx::cluster_wait();
      ptx::cluster_sync();
    }
    return;
  }

  // ---------------------------------------------------------------- consumer warps
  const int ks = warp % kWK;        // key slice of every tile
  const int nc = warp / kWK;        // query column (NT n-tiles)
  WarpState<D, NT> st;
  load_q(st, a, b, g_kv, nc, lane);
  reset_state(st);

  for (int it = 0; it < n_tiles; ++it) {
    const int s = it % STAGES;
    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
    const bool landed = ptx::mbar_wait_bounded(ptx::smem_u32(full + s), ph, a.timeout_ns, flags);
    if (!__all_sync(0xffffffffu, landed)) {   // warp-uniform decision
      if (lane == 0) raise_timeout(a, flags);
      break;
    }
    const uint32_t kbase = ptx::smem_u32(smem + s * STB);
    const uint32_t vbase = kbase + KVB;
    if constexpr (SUB == 2 && WN == 1) {
      // both of the warp's slices of the stage (tiles 0 and 1) in one step where both hold keys
      // (measured on GB300 for one warp column, up to 16 rows: the tiny workload's L2-resident step
      // 4.35 -> 4.10 us, 16 rows at 2^18 keys 90.3 -> 82.7 us; with two or four warp columns it
      // made each CTA slower, 32 rows at 19 splits 105.6 -> 144.2 us)
      const int kr[2] = {ks, kWK + ks};
      int key0[2], valid[2];
#pragma unroll
      for (int u = 0; u < 2; ++u) {
        const int64_t k0 = key_begin + (int64_t)it * SROWS + kr[u] * 16;
        key0[u] = (int)k0;
        valid[u] = (int)max((int64_t)0, min((int64_t)16, key_end - k0));
        if (valid[u] < 16) zero_masked_v<C::HALVES, C::HALVES>(smem + s * STB + KVB, kr[u], valid[u], lane, SROWS, ring);
      }
      if (valid[1] > 0)
        consume_tile2<D, NT, C::HALVES, CAUSAL, BF16>(st, kbase, vbase, valid, key0, kr, lane, a.scale_log2, SROWS,
                                                      ring);
      else if (valid[0] > 0)
        consume_tile<D, NT, C::HALVES, CAUSAL, BF16>(st, kbase, vbase, valid[0], key0[0], kr[0], lane,
                                                     a.scale_log2, SROWS, ring);
    } else {
#pragma unroll
      for (int sub = 0; sub < SUB; ++sub) {
        const int kr = sub * kWK + ks;                      // 16-key slice of the stage's box rows
        const int64_t key0 = key_begin + (int64_t)it * SROWS + kr * 16;
        const int valid = (int)max((int64_t)0, min((int64_t)16, key_end - key0));
        if (valid < 16) zero_masked_v<C::HALVES, C::HALVES>(smem + s * STB + KVB, kr, valid, lane, SROWS, ring);
        if (valid > 0)
          consume_tile<D, NT, C::HALVES, CAUSAL, BF16>(st, kbase, vbase, valid, (int)key0, kr, lane, a.scale_log2,
                                                       SROWS, ring);
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(empty + s));
  }

  // all tiles consumed (the ring is free); a wait that gave up anywhere -> leave the output alone
  if (threadIdx.x == 0) ptx::grid_launch_dependents();   // a separate merge kernel may start launching
  const bool aborted = ptx::named_bar_or(1, C::CTHREADS, flags[0] != 0);
  if constexpr (CLUSTER) {
    // push this CTA's partial of every item to the item's owner (distributed shared memory) and
    // its completion flag to every CTA; one cluster barrier; then each CTA folds the items it owns
    // from its own shared memory and leaves -- nothing reads another CTA's shared memory.  A CTA
    // whose wait gave up pushes no partial and flags it incomplete.
    using RV = ClusterRecv<C::WROWS * WN, D>;
    const uint32_t recv = ptx::smem_u32(smem + RECV_OFF);
    const int n = a.n_splits;
    ptx::cluster_wait();   // every CTA of the cluster is running: its shared memory may be written
    if (!aborted) {
      float* scratch = reinterpret_cast<float*>(smem);
      stash_warp<D, NT, WN, STAGES>(st, scratch, warp, lane, a.status);
      ptx::named_bar_sync(1, C::CTHREADS);
      push_cta_partial<D, NT, WN, STAGES>(a, scratch, recv, n, split, threadIdx.x, C::CTHREADS);
    }
    if (threadIdx.x < n)   // this CTA's flag into CTA threadIdx.x's receiving area
      ptx::st_cluster_s32(ptx::mapa(recv + RV::VALID + split * 4, threadIdx.x), aborted ? 0 : 1);
    ptx::cluster_sync();   // every push (and flag) complete and visible to its owner
    fold_received<C::WROWS * WN, D, C::CTHREADS, BF16>(a, b, g_kv, smem + RECV_OFF, n, split);
    return;
  }
  if (aborted) return;
  float* scratch = reinterpret_cast<float*>(smem);
  stash_warp<D, NT, WN, STAGES>(st, scratch, warp, lane, a.status);
  ptx::named_bar_sync(1, C::CTHREADS);
  const bool single = (a.n_splits == 1);
  emit_slice<D, NT, WN, STAGES, 1, BF16>(a, scratch, b, g_kv, split, single, threadIdx.x, C::CTHREADS);
  if (single || !a.merge_in_kernel) return;
  if (last_to_arrive<C::CTHREADS>(a, unit, a.n_splits, flags))
    merge_unit<D, NT, WN, STAGES, BF16>(a, b, g_kv, unit, a.n_splits);
}

// =====================================================================================
// paged K/V: persistent CTAs over (sequence, partition, KV head) items
// =====================================================================================
// Longest-first order of the non-empty sequences of a single-pass launch (every length <= P;
// one warp, the same result in every CTA): a stable counting sort on kSizeClasses classes of
// the length, longest class first; order[0, non-empty sequences) receives the indices.
__device__ __forceinline__ void sort_by_length(const int* lens, int N, int P, int* order, int* cls, int lane) {
  for (int c = lane; c < kSizeClasses; c += 32) cls[c] = 0;
  __syncwarp();
  auto class_of = [&](int i) {
    const int len = i < N ? lens[i] : 0;
    return len > 0 ? kSizeClasses - 1 - (int)((int64_t)(len - 1) * kSizeClasses / P) : kSizeClasses;
  };
  for (int base = 0; base < N; base += 32) {   // class sizes
    const int c = class_of(base + lane);
    const unsigned peers = __match_any_sync(0xffffffffu, c);
    if (c < kSizeClasses && lane == __ffs(peers) - 1) cls[c] += __popc(peers);
    __syncwarp();
  }
  static_assert(kSizeClasses == 64, "two classes per lane");
  const int h0 = cls[2 * lane], h1 = cls[2 * lane + 1];
  int incl = h0 + h1;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int t = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += t;
  }
  __syncwarp();
  cls[2 * lane] = incl - h0 - h1;             // first slot of each class
  cls[2 * lane + 1] = incl - h1;
  __syncwarp();
  for (int base = 0; base < N; base += 32) {   // scatter, in index order within a class
    const int i = base + lane;
    const int c = class_of(i);
    const unsigned peers = __match_any_sync(0xffffffffu, c);
    if (c < kSizeClasses) order[cls[c] + __popc(peers & ((1u << lane) - 1u))] = i;
    __syncwarp();
    if (c < kSizeClasses && lane == __ffs(peers) - 1) cls[c] += __popc(peers);
    __syncwarp();
  }
}

struct ItemDesc {
  int b, g, p, kind;        // g: first KV head of the item's group; kind: 0 partition, 2 no more items
  int n_tiles, n_parts, n_boxes, item;   // item: queue index (test hook)
  int64_t key_begin, key_end;
};
static_assert(sizeof(ItemDesc) == 48, "descriptor slot size");

// Warps: consumers 0..CONSUMERS-1, TMA producer CONSUMERS, scheduler CONSUMERS+1,
// epilogue CONSUMERS+2.
//  * scheduler: takes item indices from the queue (one at a time), maps an index to
//    (sequence, partition, group of HG KV heads) through a prefix sum of the sequences'
//    partition counts (so no index is empty; a single-pass launch takes the sequences
//    longest first), reads the partition's block
//    ids and publishes a descriptor into a kItemSlots-deep ring -- claiming an item only
//    when a slot is free.
//  * producer: for each descriptor, TMA-loads the partition's K/V blocks into the ring,
//    one box per block (or part of a block) holding the rows of all HG heads, so a box
//    moves HG times the bytes of a single head's rows.
//  * consumers: with HG heads, kWK/HG key-slice warps per head (tile = 16*kWK/HG keys);
//    with HG = 4 every warp owns one head outright.
//  * consumers: for each descriptor, the tile loop; at its end they leave their
//    (O, m, l) in one of EPI_BUFS scratch buffers and go on with the next item.
//  * epilogue: combines the consumer warps of a finished item and writes the f16
//    output (one-partition sequences) or the partition's fp32 partial; the partials
//    are folded by gqa_paged_merge_kernel (the second pass of paged attention v2).
template <int D, int NT, int WN, int STAGES, int HG, bool BF16, bool VLLM>
__global__ void __launch_bounds__(Cfg<D, NT, WN, STAGES>::PTHREADS)
gqa_paged_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const DecodeArgs a) {
  using C = Cfg<D, NT, WN, STAGES>;
  static_assert(HG == 1 || HG == 2 || HG == 4, "head group");
  static_assert(HG == 1 || WN == 1, "head groups need a single query column");
  constexpr int KS = kWK / HG;          // key-slice warps per head
  constexpr int TK = 16 * KS;           // keys per tile
  constexpr int BOXP = HG * C::HALVES;  // 64-column planes per box
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  float* scratch = reinterpret_cast<float*>(smem + C::PSCRATCH_OFF);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::PCTRL_OFF);
  uint64_t* empty = full + STAGES;
  uint64_t* ifull = empty + STAGES;
  uint64_t* iempty = ifull + kItemSlots;
  uint64_t* sfull = iempty + kItemSlots;                       // scratch buffer filled by the consumers
  uint64_t* sfree = sfull + C::EPI_BUFS;                          // scratch buffer emptied by the epilogue warp
  volatile int* flags = reinterpret_cast<volatile int*>(sfree + C::EPI_BUFS);  // [0] abort
  ItemDesc* desc = reinterpret_cast<ItemDesc*>(const_cast<int*>(flags + 4));
  ItemDesc* edesc = desc + kItemSlots;                          // item of each scratch buffer
  int* boxy = reinterpret_cast<int*>(edesc + C::EPI_BUFS);      // [kItemSlots][kMaxBoxesPerPart] box rows
  int* pre = boxy + kItemSlots * kMaxBoxesPerPart;              // [N + 1] partition-count prefix
  int* lens_s = pre + kPagedSeqs + 1;                           // [N] clamped lengths
  int* order = lens_s + kPagedSeqs;                             // [N] single pass: sequences, longest first
  int* cls = order + kPagedSeqs;                                // [kSizeClasses] counting-sort cursors

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int P = a.partition_size;
  const int N = a.B;
  const int cap = min(a.max_blocks_per_seq * a.block_size, a.n_splits * P);
  const Win ring{ptx::smem_u32(smem), ptx::smem_u32(smem) + (uint32_t)C::PIPE_BYTES, a.status};
  // the per-sequence tables in shared memory hold kPagedSeqs entries (the host splits larger batches)
  if (!idx_ok(N, kPagedSeqs + 1, a.status)) return;

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(full + s), 1);
      ptx::mbar_init(ptx::smem_u32(empty + s), C::CONSUMERS);
    }
    for (int s = 0; s < kItemSlots; ++s) {
      ptx::mbar_init(ptx::smem_u32(ifull + s), 1);
      ptx::mbar_init(ptx::smem_u32(iempty + s), C::CONSUMERS + 1);
    }
    for (int s = 0; s < C::EPI_BUFS; ++s) {
      ptx::mbar_init(ptx::smem_u32(sfull + s), C::CONSUMERS);
      ptx::mbar_init(ptx::smem_u32(sfree + s), 1);
    }
    flags[0] = 0;
    flags[1] = 0;
    pre[0] = 0;
    ptx::fence_mbar_init();
  }
  // launched as a programmatic dependent: nothing in global memory is read or written before the
  // previous kernel in the stream has completed
  ptx::grid_dependency_wait();
  // lengths (clamped to what the table can hold) and partitions per sequence
  for (int i = threadIdx.x; i < N; i += blockDim.x) {
    int len = __ldg(a.seq_lens + i);
    if (len < 0 || len > cap) {
      if (blockIdx.x == 0) atomicOr(a.status, kDevBadInput);
      len = len < 0 ? 0 : cap;
    }
    lens_s[i] = len;
    pre[i + 1] = (len + P - 1) / P;
  }
  __syncthreads();
  if (warp == 0) {   // inclusive scan of pre[1..N], 32 entries at a time
    int carry = 0;
    for (int base = 0; base < N; base += 32) {
      const int i = base + lane;
      int v = i < N ? pre[i + 1] : 0;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += t;
      }
      if (i < N) pre[i + 1] = v + carry;
      carry += __shfl_sync(0xffffffffu, v, 31);
    }
  }
  if (warp == C::CONSUMERS && lane == 0) {
    ptx::prefetch_tensormap(&tmK);
    ptx::prefetch_tensormap(&tmV);
  }
  __syncthreads();
  const int groups = a.h_kv / HG;
  const int64_t total = (int64_t)pre[N] * groups;
  const int br = min(a.block_size, TK);  // rows per box
  // sequences without keys get zero output rows (spread over the CTAs)
  for (int b = blockIdx.x; b < N; b += gridDim.x) {
    if (lens_s[b] != 0 || !idx_ok((int64_t)(b + 1) * a.T_q * a.h_q - 1, a.R, a.status)) continue;
    __half* dst = a.o + (int64_t)b * a.T_q * a.h_q * D;
    for (int i = threadIdx.x; i < a.T_q * a.h_q * D; i += blockDim.x) dst[i] = __float2half_rn(0.f);
  }

  // ---------------------------------------------------------------- epilogue warp
  if (warp == C::CONSUMERS + 2) {
    for (int ke = 0;; ++ke) {
      const int buf = ke % C::EPI_BUFS;
      const bool got = ptx::mbar_wait_bounded(ptx::smem_u32(sfull + buf), (uint32_t)(ke / C::EPI_BUFS) & 1u,
                                              a.timeout_ns, flags);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0) raise_timeout(a, flags);
        break;
      }
      const ItemDesc d = edesc[buf];
      if (d.kind == 2) break;
      const float* sb = reinterpret_cast<const float*>(smem + C::PSCRATCH_OFF + buf * C::PSCRATCH_STRIDE);
      emit_slice_warp<D, NT, WN, STAGES, HG, BF16>(a, sb, d.b, d.g, d.p, d.n_parts == 1, lane);
      __syncwarp();
      if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(sfree + buf));
    }
    if (lane == 0) ptx::grid_launch_dependents();   // the merge pass may start launching
    return;
  }

  // ---------------------------------------------------------------- scheduler warp
  if (warp == C::CONSUMERS + 1) {
    bool sorted = false;
    for (int k = 0;; ++k) {
      const int slot = k % kItemSlots;
      int ok = 1;
      if (lane == 0 && k >= kItemSlots)
        ok = ptx::mbar_wait_bounded(ptx::smem_u32(iempty + slot), ((uint32_t)(k / kItemSlots) & 1u) ^ 1u,
                                    a.timeout_ns, flags) ? 1 : 0;
      if (__shfl_sync(0xffffffffu, ok, 0) == 0) {
        if (lane == 0) raise_timeout(a, flags);
        break;
      }
      // claim the next item only once a slot is free: items claimed early are work this CTA
      // holds back from the others at the end of the queue
      uint32_t it = 0;
      if (lane == 0) it = atomicAdd(a.queue, 1u);
      it = __shfl_sync(0xffffffffu, it, 0);
      ItemDesc d;
      d.kind = 2;
      d.b = d.g = d.p = d.n_tiles = d.n_parts = d.n_boxes = 0;
      d.item = (int)it;
      d.key_begin = d.key_end = 0;
      if ((int64_t)it < total) {
        d.g = (int)(it % (uint32_t)groups) * HG;
        const int j = (int)(it / (uint32_t)groups);
        if (a.n_splits > 1) {
          int lo = 0, hi = N;                        // pre[lo] <= j < pre[hi]
          while (hi - lo > 1) {
            const int mid = (lo + hi) >> 1;
            if (pre[mid] <= j) lo = mid; else hi = mid;
          }
          d.b = lo;
          d.p = j - pre[lo];
        } else {
          // single pass: sequences longest first, so that the queue ends with its shortest items
          if (!sorted) {
            sort_by_length(lens_s, N, P, order, cls, lane);
            sorted = true;
          }
          d.b = order[j];
          d.p = 0;
        }
        d.n_parts = (lens_s[d.b] + P - 1) / P;
        d.kind = 0;
        d.key_begin = (int64_t)d.p * P;
        d.key_end = min(d.key_begin + P, (int64_t)lens_s[d.b]);
        d.n_tiles = (int)((d.key_end - d.key_begin + TK - 1) / TK);
        d.n_boxes = (int)((d.key_end - d.key_begin + br - 1) / br);
        // pool row of every box of the partition (-1: block id outside the pool, not loaded),
        // so that the producer thread only reads them
        const int bs = a.block_size;
        const int32_t* row = a.block_tables + (int64_t)d.b * a.max_blocks_per_seq + d.key_begin / bs;
        int* dst = boxy + slot * kMaxBoxesPerPart;
        for (int i = lane; i < d.n_boxes; i += 32) {
          const int rel = i * br;                   // key offset in the partition (block aligned start)
          const int blk = rel / bs;
          // the entry lies in sequence d.b's row of the table, the box in this slot's list
          if (!idx_ok(d.b, N, a.status) || !idx_ok(d.key_begin / bs + blk, a.max_blocks_per_seq, a.status) ||
              !idx_ok(i, kMaxBoxesPerPart, a.status)) {
            if (i < kMaxBoxesPerPart) dst[i] = -1;
            continue;
          }
          int id = __ldg(row + blk);
          if (id < 0 || id >= a.num_blocks) {
            atomicOr(a.status, kDevBadInput);
            id = -1;
          }
          dst[i] = id < 0 ? -1 : id * bs + (rel - blk * bs);
        }
      }
      __threadfence_block();
      __syncwarp();
      if (lane == 0) {
        desc[slot] = d;
        ptx::mbar_arrive(ptx::smem_u32(ifull + slot));
      }
      if (d.kind == 2) break;
    }
    return;
  }

  // ---------------------------------------------------------------- TMA producer warp
  if (warp == C::CONSUMERS) {
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_first();
      const int nbox = TK / br;   // boxes per tile
      const int bs_shift = __ffs(a.block_size) - 1;   // block sizes are powers of two
      int tile_it = 0, stall_tile = -1;
      bool gave_up = false;
      for (int k = 0;; ++k) {
        const int slot = k % kItemSlots;
        if (!ptx::mbar_wait_bounded(ptx::smem_u32(ifull + slot), (uint32_t)(k / kItemSlots) & 1u, a.timeout_ns,
                                    flags)) {
          raise_timeout(a, flags);
          gave_up = true;
          break;
        }
        const ItemDesc d = desc[slot];
        if (d.kind == 2) break;
        // test hook: the second tile of queue item stall_cta is never loaded
        if (a.stall_cta >= 0 && d.item == a.stall_cta && d.n_tiles > 1) stall_tile = tile_it + 1;
        const int* by = boxy + slot * kMaxBoxesPerPart;
        for (int t = 0; t < d.n_tiles; ++t, ++tile_it) {
          const int s = tile_it % STAGES;
          const uint32_t ph = (uint32_t)(tile_it / STAGES) & 1u;
          if (tile_it >= STAGES &&
              !ptx::mbar_wait_bounded(ptx::smem_u32(empty + s), ph ^ 1u, a.timeout_ns, flags)) {
            raise_timeout(a, flags);
            gave_up = true;
            break;
          }
          if (tile_it == stall_tile) continue;
          const uint32_t kdst = ptx::smem_u32(smem + s * C::STAGE_BYTES);
          const uint32_t vdst = kdst + C::KV_BYTES;
          const uint32_t fb = ptx::smem_u32(full + s);
          // box j of tile t holds keys [(t*nbox + j)*br, +br) of the partition
          const int b0 = t * nbox;
          const int nb_t = min(nbox, d.n_boxes - b0);
          // a box is loaded when its pool row is valid -- and, checked, when the box and its
          // destination are in range
          auto box_ok = [&](int j) {
            if (!idx_ok(b0 + j, kMaxBoxesPerPart, a.status)) return false;
            const int y = by[b0 + j];
            if (y < 0) return false;
            const uint32_t off = j * br * 128 * BOXP;
            if (!smem_ok(kdst + off, br * 128 * BOXP, ring.lo, ring.hi, a.status) ||
                !smem_ok(vdst + off, br * 128 * BOXP, ring.lo, ring.hi, a.status))
              return false;
            if constexpr (VLLM) {
              return idx_ok((int64_t)(y >> bs_shift) * a.h_kv + d.g + HG - 1, (int64_t)a.num_blocks * a.h_kv,
                            a.status);
            } else {
              return idx_ok(y, (int64_t)a.num_blocks * a.block_size, a.status) &&
                     idx_ok(d.g + HG - 1, a.h_kv, a.status);
            }
          };
          int n_load = 0;
          for (int j = 0; j < nb_t; ++j) n_load += box_ok(j) ? 1 : 0;
          ptx::mbar_arrive_expect_tx(fb, (uint32_t)(n_load * br * 128 * 2 * BOXP));
          for (int j = 0; j < nb_t; ++j) {
            if (!box_ok(j)) continue;
            const int y = by[b0 + j];
            const uint32_t off = j * br * 128 * BOXP;
            if constexpr (VLLM) {
              // pool row y = block * block_size (boxes are whole blocks): both boxes start at head
              // block*h_kv + g of the (block, head)-major caches
              const int kvh = (y >> bs_shift) * a.h_kv + d.g;
              ptx::tma_load_4d(kdst + off, &tmK, fb, 0, 0, 0, kvh, pol);
              ptx::tma_load_3d(vdst + off, &tmV, fb, 0, 0, kvh, pol);
            } else {
              ptx::tma_load_3d(kdst + off, &tmK, fb, 0, y, d.g * C::HALVES, pol);
              ptx::tma_load_3d(vdst + off, &tmV, fb, 0, y, d.g * C::HALVES, pol);
            }
          }
        }
        ptx::mbar_arrive(ptx::smem_u32(iempty + slot));
        if (gave_up) break;
      }
      if (gave_up || stall_tile >= 0) {
        // wait (bounded) for copies still in flight before the CTA can exit
        for (int it = max(0, tile_it - STAGES); it < tile_it; ++it) {
          if (it == stall_tile) continue;
          ptx::mbar_wait_bounded(ptx::smem_u32(full + (it % STAGES)), (uint32_t)(it / STAGES) & 1u,
                                 a.timeout_ns, nullptr);
        }
      }
    }
    return;
  }

  // ---------------------------------------------------------------- consumer warps
  const int hh = HG > 1 ? warp / KS : 0;           // head within the item's group
  const int ks = HG > 1 ? warp % KS : warp % kWK;  // key slice of every tile
  const int nc = HG > 1 ? 0 : warp / kWK;          // query column
  const int head_off = hh * C::HALVES * br * 128;  // first plane of this warp's head in a box
  WarpState<D, NT> st;
  int tile_it = 0, kc = 0;   // tiles consumed, items handed to the epilogue warp
  for (int k = 0;; ++k) {
    const int slot = k % kItemSlots;
    const bool got = ptx::mbar_wait_bounded(ptx::smem_u32(ifull + slot), (uint32_t)(k / kItemSlots) & 1u,
                                            a.timeout_ns, flags);
    const bool ok_w = __all_sync(0xffffffffu, got);
    if (!ok_w && lane == 0) raise_timeout(a, flags);
    if (ptx::named_bar_or(1, C::CTHREADS, !ok_w)) return;          // every consumer warp leaves together
    const ItemDesc d = desc[slot];
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(iempty + slot));
    bool aborted = false;
    if (d.kind != 2) {
      load_q(st, a, d.b, d.g + hh, nc, lane);
      reset_state(st);
      for (int t = 0; t < d.n_tiles; ++t, ++tile_it) {
        const int s = tile_it % STAGES;
        const uint32_t ph = (uint32_t)(tile_it / STAGES) & 1u;
        const bool landed = ptx::mbar_wait_bounded(ptx::smem_u32(full + s), ph, a.timeout_ns, flags);
        if (!__all_sync(0xffffffffu, landed)) {
          if (lane == 0) raise_timeout(a, flags);
          aborted = true;
          break;
        }
        const uint32_t kbase = ptx::smem_u32(smem + s * C::STAGE_BYTES) + head_off;
        const uint32_t vbase = kbase + C::KV_BYTES;
        const int64_t key0 = d.key_begin + (int64_t)t * TK + ks * 16;
        const int valid = (int)max((int64_t)0, min((int64_t)16, d.key_end - key0));
        if (valid < 16) {
          uint8_t* vh = smem + s * C::STAGE_BYTES + C::KV_BYTES + head_off;
          if constexpr (VLLM) {
            zero_masked_v_vllm<D>(vh, ks, valid, lane, br, br * 128 * BOXP, ring);
          } else {
            zero_masked_v<C::HALVES, BOXP>(vh, ks, valid, lane, br, ring);
          }
        }
        if (valid > 0)
          consume_tile<D, NT, BOXP, false, BF16, VLLM>(st, kbase, vbase, valid, (int)key0, ks, lane, a.scale_log2,
                                                       br, ring);
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(empty + s));
      }
    }
    // hand the item (or the end marker) to the epilogue warp through scratch buffer kc % C::EPI_BUFS
    const int buf = kc % C::EPI_BUFS;
    bool free_ok = true;
    if (!aborted && kc >= C::EPI_BUFS)
      free_ok = ptx::mbar_wait_bounded(ptx::smem_u32(sfree + buf), ((uint32_t)(kc / C::EPI_BUFS) & 1u) ^ 1u,
                                       a.timeout_ns, flags);
    if (!__all_sync(0xffffffffu, free_ok)) {
      if (lane == 0) raise_timeout(a, flags);
      aborted = true;
    }
    // every consumer warp reaches this barrier once per item, aborted or not
    if (ptx::named_bar_or(1, C::CTHREADS, aborted || flags[0] != 0)) return;
    if (d.kind != 2) {
      float* sb = reinterpret_cast<float*>(smem + C::PSCRATCH_OFF + buf * C::PSCRATCH_STRIDE);
      stash_warp<D, NT, WN, STAGES>(st, sb, warp, lane, a.status);
    }
    if (warp == 0 && lane == 0) edesc[buf] = d;
    __threadfence_block();
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(sfull + buf));
    ++kc;
    if (d.kind == 2) break;
  }
  // the last CTA to finish resets the item queue for the next launch
  __threadfence();
  ptx::named_bar_sync(1, C::CTHREADS);
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(a.done, 1u);
    if (prev == gridDim.x - 1) {
      atomicExch(a.queue, 0u);
      atomicExch(a.done, 0u);
    }
  }
}

// Every decode kernel is launched with programmatic stream serialisation: its CTAs may begin (and
// set up their barriers and tensor memory) while the previous kernel in the stream finishes, and
// wait in griddepcontrol.wait before they touch global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_dependent(void (*kernel)(KArgs...), dim3 grid, unsigned block, unsigned smem, cudaStream_t st,
                             dim3 cluster, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = dim3(block, 1, 1);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  int n = 1;
  if (cluster.x * cluster.y * cluster.z > 1) {
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = cluster.x;
    attr[1].val.clusterDim.y = cluster.y;
    attr[1].val.clusterDim.z = cluster.z;
    n = 2;
  }
  cfg.attrs = attr;
  cfg.numAttrs = n;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

}  // namespace gqa
