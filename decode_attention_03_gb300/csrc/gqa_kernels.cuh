// Split-KV GQA decode kernels for sm_103a.
//
// One CTA handles one (sequence b, KV head g, split) work unit: the G*T_q query
// rows that share KV head g, against one contiguous slice of the key axis.
// Page "kernbench2 ... _gqa_attention_decode_long.py" ("GQA fused-attention
// decode kernel -- long context") describes the same decomposition for a PE
// mesh: every rank sweeps its S_kv slice in tiles, keeps a running (m, l, O)
// and merges partials with _merge_running; here the ranks become CTAs and the
// reduce-to-root becomes the last-arriving CTA of the unit merging all splits.
// The paged variant follows page "muh_kernel_map.py", VLLM_KERNEL_MAP
// 'paged_attention_v2' (per-partition pass, then a cross-partition merge).
//
// CTA layout: kWK*WN consumer warps + 1 producer warp.
//  * producer (one lane): TMA 2-D tensor loads of each 64-key K and V tile
//    (128-byte swizzled boxes of 64 f16 columns) into a STAGES-deep ring of
//    shared-memory buffers, signalled through mbarriers (full/empty).
//  * consumer warp (ks, nc): keys [16*ks, 16*ks+16) of every tile, query
//    n-tiles [nc*NT, nc*NT+NT) (8 query rows each).  Scores are computed
//    transposed, S^T = K Q^T (keys on the MMA's M side, so G*T_q = 4 wastes
//    only half of an n=8 tile), the softmax runs in the accumulator layout, P
//    is transposed in registers (movmatrix) into the B operand of
//    O^T += V^T P^T.  Each warp keeps its own running (m, l, O) over its keys;
//    the warps' states are merged through shared memory at the end.
#pragma once
#include <cuda.h>
#include <cuda_fp16.h>
#include <math_constants.h>
#include <stdint.h>

#include "ptx.cuh"

namespace gqa {

constexpr int kWK = 4;             // consumer warps along the key axis
constexpr int kTile = 16 * kWK;    // keys per pipeline stage
constexpr uint32_t kDevTimeout = 1u;
constexpr uint32_t kDevBadInput = 2u;
constexpr float kLn2 = 0.6931471805599453f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxPagedBlocksPerPart = 512;

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
  // paged
  const int32_t* block_tables;
  const int32_t* seq_lens;
  int max_blocks_per_seq;
  int num_blocks;
  int block_size;
  int partition_size;
  // shape
  int B, T_q, h_q, h_kv, G, rows;  // rows = G*T_q query rows per unit
  int64_t R;                        // B*T_q*h_q rows of the output
  int64_t S_kv;                     // contiguous: keys per sequence
  int64_t s_begin, s_len;           // contiguous: key range swept
  int n_splits;                     // contiguous: splits per unit; paged: max partitions
  int merge_in_kernel;              // last CTA of a unit merges the splits
  float scale_log2;                 // scale * log2(e)
  uint64_t timeout_ns;
  int stall_cta;                    // test hook: CTA whose producer withholds tile 1 (-1 none)
};

template <int D, int NT, int WN, int STAGES>
struct Cfg {
  static constexpr int HALVES = D / 64;
  static constexpr int HALF_BYTES = kTile * 128;         // [kTile][64] f16, 128B-swizzled
  static constexpr int KV_BYTES = HALVES * HALF_BYTES;   // one K (or V) tile
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int CONSUMERS = kWK * WN;
  static constexpr int THREADS = (CONSUMERS + 1) * 32;
  static constexpr int WROWS = 8 * NT;                   // query rows per consumer warp
  static constexpr int OSTRIDE = D + 4;                  // padded row of the merge scratch
  static constexpr int WSCRATCH = WROWS * (OSTRIDE + 2); // floats per warp
  static constexpr int SCRATCH_BYTES = CONSUMERS * WSCRATCH * 4;
  static constexpr int PIPE_BYTES = STAGES * STAGE_BYTES;
  static constexpr int DATA_BYTES = PIPE_BYTES > SCRATCH_BYTES ? PIPE_BYTES : SCRATCH_BYTES;
  static constexpr int CTRL_BYTES = 2 * STAGES * 8 + 16 + kMaxPagedBlocksPerPart * 4;
  static constexpr int SMEM_BYTES = 1024 + DATA_BYTES + CTRL_BYTES;
};

// Row r of a unit (0 <= r < G*T_q) is query token r / G, head g*G + r % G.
__device__ __forceinline__ int64_t out_row(const DecodeArgs& a, int b, int g, int r) {
  const int tq = r / a.G, hh = r - tq * a.G;
  return ((int64_t)b * a.T_q + tq) * a.h_q + (int64_t)g * a.G + hh;
}

// Address of 16-byte chunk c (of D/8) of row `row` in a [kTile][D] tile stored
// as D/64 swizzled [kTile][64] boxes.
template <int HALF_BYTES>
__device__ __forceinline__ uint32_t tile_addr(uint32_t base, int row, int c) {
  return base + (c >> 3) * HALF_BYTES + row * 128 + ((((c & 7) ^ (row & 7))) << 4);
}

// Merge n partials of one output row element; weights exp(m_s - M).
// Empty partials (m = -inf) contribute nothing; all empty -> (M=-inf, L=0, O=0).

template <int D, int NT, int WN, int STAGES, bool PAGED>
__global__ void __launch_bounds__(Cfg<D, NT, WN, STAGES>::THREADS)
gqa_split_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                 const DecodeArgs a) {
  using C = Cfg<D, NT, WN, STAGES>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::DATA_BYTES);
  uint64_t* empty = full + STAGES;
  volatile int* flags = reinterpret_cast<volatile int*>(empty + STAGES);  // [0] abort, [1] last-CTA
  int* blk_ids = const_cast<int*>(reinterpret_cast<volatile int*>(flags + 4));

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g_kv = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
  const int unit = b * a.h_kv + g_kv;

  // ---- this CTA's key range [key_begin, key_end) and the number of splits of its unit
  int64_t key_begin, key_end, y_base = 0;
  int n_tiles, n_split_unit;
  if constexpr (!PAGED) {
    const int64_t tiles_total = (a.s_len + kTile - 1) / kTile;
    const int64_t t0 = tiles_total * split / a.n_splits;
    const int64_t t1 = tiles_total * (split + 1) / a.n_splits;
    key_begin = a.s_begin + t0 * kTile;
    key_end = min(a.s_begin + t1 * kTile, a.s_begin + a.s_len);
    n_tiles = (int)(t1 - t0);
    n_split_unit = a.n_splits;
    y_base = (int64_t)b * a.S_kv;
  } else {
    int len = __ldg(a.seq_lens + b);
    const int cap = min(a.max_blocks_per_seq * a.block_size, a.n_splits * a.partition_size);
    if (len < 0 || len > cap) {
      if (threadIdx.x == 0 && split == 0) atomicOr(a.status, kDevBadInput);
      len = len < 0 ? 0 : cap;
    }
    n_split_unit = (len + a.partition_size - 1) / a.partition_size;
    if (split >= n_split_unit) {
      if (split == 0) {  // empty sequence: its output rows are zero
        for (int i = threadIdx.x; i < a.rows * D; i += blockDim.x) {
          const int r = i / D, d = i - r * D;
          a.o[out_row(a, b, g_kv, r) * D + d] = __float2half_rn(0.f);
        }
      }
      return;
    }
    key_begin = (int64_t)split * a.partition_size;
    key_end = min(key_begin + a.partition_size, (int64_t)len);
    n_tiles = (int)((key_end - key_begin + kTile - 1) / kTile);
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(full + s), 1);
      ptx::mbar_init(ptx::smem_u32(empty + s), C::CONSUMERS);
    }
    flags[0] = 0;
    flags[1] = 0;
    ptx::fence_mbar_init();
  }
  if constexpr (PAGED) {
    // block ids of this partition, read once (coalesced) by the producer warp
    if (warp == C::CONSUMERS) {
      const int nb = (int)((key_end - key_begin + a.block_size - 1) / a.block_size);
      const int first = (int)(key_begin / a.block_size);
      const int32_t* row = a.block_tables + (int64_t)b * a.max_blocks_per_seq + first;
      for (int i = lane; i < nb; i += 32) {
        int id = __ldg(row + i);
        if (id < 0 || id >= a.num_blocks) {
          atomicOr(a.status, kDevBadInput);
          id = -1;
        }
        blk_ids[i] = id;
      }
    }
  }
  if (warp == C::CONSUMERS && lane == 0) {
    ptx::prefetch_tensormap(&tmK);
    ptx::prefetch_tensormap(&tmV);
  }
  __syncthreads();

  // =====================================================================
  // producer warp
  // =====================================================================
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
        if (it >= STAGES) {
          if (!ptx::mbar_wait_bounded(ptx::smem_u32(empty + s), ph ^ 1u, a.timeout_ns, flags)) {
            atomicOr(a.status, kDevTimeout);
            flags[0] = 1;
            gave_up = true;
            break;
          }
        }
        issued = it + 1;
        if (it == stall_tile) continue;  // test hook: this tile is never loaded
        const uint32_t kdst = ptx::smem_u32(smem + s * C::STAGE_BYTES);
        const uint32_t vdst = kdst + C::KV_BYTES;
        const uint32_t fb = ptx::smem_u32(full + s);
        if constexpr (!PAGED) {
          ptx::mbar_arrive_expect_tx(fb, C::STAGE_BYTES);
          const int y = (int)(y_base + key_begin + (int64_t)it * kTile);
#pragma unroll
          for (int h = 0; h < C::HALVES; ++h) {
            const int x = g_kv * D + h * 64;
            ptx::tma_load_2d(kdst + h * C::HALF_BYTES, &tmK, fb, x, y, pol);
            ptx::tma_load_2d(vdst + h * C::HALF_BYTES, &tmV, fb, x, y, pol);
          }
        } else {
          const int bs = a.block_size;
          const int64_t k0 = key_begin + (int64_t)it * kTile;
          const int nblk_tile = kTile / bs;
          const int first = (int)((k0 - key_begin) / bs);
          int n_load = 0;
          for (int j = 0; j < nblk_tile; ++j) {
            if (k0 + (int64_t)j * bs < key_end && blk_ids[first + j] >= 0) ++n_load;
          }
          ptx::mbar_arrive_expect_tx(fb, (uint32_t)(n_load * bs * 128 * 2 * C::HALVES));
          for (int j = 0; j < nblk_tile; ++j) {
            if (k0 + (int64_t)j * bs >= key_end) break;
            const int id = blk_ids[first + j];
            if (id < 0) continue;
            const int y = id * bs;
#pragma unroll
            for (int h = 0; h < C::HALVES; ++h) {
              const int x = g_kv * D + h * 64;
              const uint32_t off = h * C::HALF_BYTES + j * bs * 128;
              ptx::tma_load_2d(kdst + off, &tmK, fb, x, y, pol);
              ptx::tma_load_2d(vdst + off, &tmV, fb, x, y, pol);
            }
          }
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
    return;
  }

  // =====================================================================
  // consumer warps
  // =====================================================================
  const int ks = warp % kWK;        // key slice of every tile
  const int nc = warp / kWK;        // query column (NT n-tiles)
  const int gq = lane >> 2, tq4 = lane & 3;
  constexpr int KD = D / 16;        // k-steps over d (QK) / m-tiles over d (PV)

  // Q^T fragments (B operand of S^T = K Q^T): b0 = Q[row gq][16kk + 2tq4 ..+1], b1 = +8
  uint32_t qf[NT][KD][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    const int r = (nc * NT + nt) * 8 + gq;
    if (r < a.rows) {
      const uint32_t* qp = reinterpret_cast<const uint32_t*>(a.q + out_row(a, b, g_kv, r) * D);
#pragma unroll
      for (int kk = 0; kk < KD; ++kk) {
        qf[nt][kk][0] = __ldg(qp + kk * 8 + tq4);
        qf[nt][kk][1] = __ldg(qp + kk * 8 + 4 + tq4);
      }
    } else {
#pragma unroll
      for (int kk = 0; kk < KD; ++kk) qf[nt][kk][0] = qf[nt][kk][1] = 0u;
    }
  }

  float acc[KD][NT][4];
#pragma unroll
  for (int i = 0; i < KD; ++i)
#pragma unroll
    for (int nt = 0; nt < NT; ++nt)
#pragma unroll
      for (int c = 0; c < 4; ++c) acc[i][nt][c] = 0.f;
  float m_run[NT][2], l_run[NT][2];
#pragma unroll
  for (int nt = 0; nt < NT; ++nt) {
    m_run[nt][0] = m_run[nt][1] = -CUDART_INF_F;
    l_run[nt][0] = l_run[nt][1] = 0.f;
  }

  // per-lane ldmatrix row/chunk (K: non-transposed A of S^T; V: transposed A of O^T)
  const int k_row = ks * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
  const int k_c0 = lane >> 4;
  const int v_row = ks * 16 + (lane & 7) + ((lane >> 4) & 1) * 8;
  const int v_c0 = (lane >> 3) & 1;

  for (int it = 0; it < n_tiles; ++it) {
    const int s = it % STAGES;
    const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
    const bool landed = ptx::mbar_wait_bounded(ptx::smem_u32(full + s), ph, a.timeout_ns, flags);
    if (!__all_sync(0xffffffffu, landed)) {   // warp-uniform decision
      if (lane == 0) {
        atomicOr(a.status, kDevTimeout);
        flags[0] = 1;
      }
      break;
    }
    const uint32_t kbase = ptx::smem_u32(smem + s * C::STAGE_BYTES);
    const uint32_t vbase = kbase + C::KV_BYTES;
    const int64_t key0 = key_begin + (int64_t)it * kTile + ks * 16;
    const int valid = (int)max((int64_t)0, min((int64_t)16, key_end - key0));

    if (valid < 16) {
      // keys past the range: zero their V rows so that 0 * (stale or NaN) cannot reach O
      uint4* vrow = reinterpret_cast<uint4*>(smem + s * C::STAGE_BYTES + C::KV_BYTES);
      for (int i = lane; i < (16 - valid) * 8 * C::HALVES; i += 32) {
        const int h = i / ((16 - valid) * 8);
        const int rem = i - h * ((16 - valid) * 8);
        const int row = ks * 16 + valid + rem / 8;
        vrow[(h * C::HALF_BYTES + row * 128) / 16 + (rem & 7)] = make_uint4(0u, 0u, 0u, 0u);
      }
      ptx::fence_proxy_async_smem();
      __syncwarp();
    }

    if (valid > 0) {
      // ---- S^T = K Q^T : 16 keys x 8*NT query rows, fp32
      float sc[NT][4];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) sc[nt][0] = sc[nt][1] = sc[nt][2] = sc[nt][3] = 0.f;
#pragma unroll
      for (int kk = 0; kk < KD; ++kk) {
        uint32_t af[4];
        ptx::ldmatrix_x4(af, tile_addr<C::HALF_BYTES>(kbase, k_row, kk * 2 + k_c0));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) ptx::mma_16816(sc[nt], af, qf[nt][kk]);
      }
      // ---- scale (log2 domain), mask, online softmax.  sc[nt][c]: key gq (c<2) or gq+8,
      //      query row 2*tq4 + (c&1) of n-tile nt
      float alpha[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const int key = gq + ((c >> 1) << 3);
          sc[nt][c] = key < valid ? sc[nt][c] * a.scale_log2 : -CUDART_INF_F;
        }
#pragma unroll
        for (int j = 0; j < 2; ++j) {
          float mx = fmaxf(sc[nt][j], sc[nt][j + 2]);
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
          mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
          const float m_new = fmaxf(m_run[nt][j], mx);
          const float m_use = m_new == -CUDART_INF_F ? 0.f : m_new;
          alpha[nt][j] = ptx::ex2(m_run[nt][j] - m_use);
          m_run[nt][j] = m_new;
          const float p0 = ptx::ex2(sc[nt][j] - m_use);
          const float p1 = ptx::ex2(sc[nt][j + 2] - m_use);
          l_run[nt][j] = l_run[nt][j] * alpha[nt][j] + (p0 + p1);
          sc[nt][j] = p0;
          sc[nt][j + 2] = p1;
        }
      }
      // ---- rescale O^T (rows d, columns = query rows 2*tq4, 2*tq4+1)
#pragma unroll
      for (int i = 0; i < KD; ++i)
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) {
          acc[i][nt][0] *= alpha[nt][0];
          acc[i][nt][1] *= alpha[nt][1];
          acc[i][nt][2] *= alpha[nt][0];
          acc[i][nt][3] *= alpha[nt][1];
        }
      // ---- P^T as the B operand (keys x query rows): transpose 8x8 f16 blocks in registers
      uint32_t pf[NT][2];
#pragma unroll
      for (int nt = 0; nt < NT; ++nt) {
        pf[nt][0] = ptx::movmatrix_trans(ptx::pack_half2(sc[nt][0], sc[nt][1]));
        pf[nt][1] = ptx::movmatrix_trans(ptx::pack_half2(sc[nt][2], sc[nt][3]));
      }
      // ---- O^T += V^T P^T
#pragma unroll
      for (int i = 0; i < KD; ++i) {
        uint32_t af[4];
        ptx::ldmatrix_x4_trans(af, tile_addr<C::HALF_BYTES>(vbase, v_row, i * 2 + v_c0));
#pragma unroll
        for (int nt = 0; nt < NT; ++nt) ptx::mma_16816(acc[i][nt], af, pf[nt]);
      }
    }
    __syncwarp();
    if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(empty + s));
  }

  // ---- merge the kWK key-slice warps of each query column through shared memory
  constexpr uint32_t kConsumerThreads = C::CONSUMERS * 32;
  // all tiles consumed (the ring is free); a wait that gave up anywhere -> leave the output alone
  if (ptx::named_bar_or(1, kConsumerThreads, flags[0] != 0)) return;

#pragma unroll
  for (int nt = 0; nt < NT; ++nt)
#pragma unroll
    for (int j = 0; j < 2; ++j) {
      float l = l_run[nt][j];
      l += __shfl_xor_sync(0xffffffffu, l, 4);
      l += __shfl_xor_sync(0xffffffffu, l, 8);
      l += __shfl_xor_sync(0xffffffffu, l, 16);
      l_run[nt][j] = l;
    }
  float* scratch = reinterpret_cast<float*>(smem);
  {
    float* wsp = scratch + warp * C::WSCRATCH;
    float* wm = wsp + C::WROWS * C::OSTRIDE;
    float* wl = wm + C::WROWS;
#pragma unroll
    for (int nt = 0; nt < NT; ++nt) {
      const int r0 = nt * 8 + 2 * tq4;
#pragma unroll
      for (int i = 0; i < KD; ++i) {
        wsp[r0 * C::OSTRIDE + i * 16 + gq] = acc[i][nt][0];
        wsp[(r0 + 1) * C::OSTRIDE + i * 16 + gq] = acc[i][nt][1];
        wsp[r0 * C::OSTRIDE + i * 16 + gq + 8] = acc[i][nt][2];
        wsp[(r0 + 1) * C::OSTRIDE + i * 16 + gq + 8] = acc[i][nt][3];
      }
      if (gq == 0) {
        wm[r0] = m_run[nt][0];
        wm[r0 + 1] = m_run[nt][1];
        wl[r0] = l_run[nt][0];
        wl[r0 + 1] = l_run[nt][1];
      }
    }
  }
  ptx::named_bar_sync(1, kConsumerThreads);

  const bool single = (n_split_unit == 1);
  for (int idx = threadIdx.x; idx < a.rows * D; idx += kConsumerThreads) {
    const int r = idx / D, d = idx - r * D;
    const int col = r / C::WROWS, lr = r - col * C::WROWS;
    float mk[kWK];
    float M = -CUDART_INF_F;
#pragma unroll
    for (int k = 0; k < kWK; ++k) {
      const float* wsp = scratch + (col * kWK + k) * C::WSCRATCH;
      mk[k] = wsp[C::WROWS * C::OSTRIDE + lr];
      M = fmaxf(M, mk[k]);
    }
    float L = 0.f, O = 0.f;
    if (M != -CUDART_INF_F) {
#pragma unroll
      for (int k = 0; k < kWK; ++k) {
        const float* wsp = scratch + (col * kWK + k) * C::WSCRATCH;
        const float w = ptx::ex2(mk[k] - M);
        L += w * wsp[C::WROWS * C::OSTRIDE + C::WROWS + lr];
        O += w * wsp[lr * C::OSTRIDE + d];
      }
    }
    const int64_t orow = out_row(a, b, g_kv, r);
    if (single) {
      if (a.o != nullptr) {
        a.o[orow * D + d] = __float2half_rn(L > 0.f ? O / L : 0.f);
      } else {
        if (d == 0) {
          a.m_out[orow] = M * kLn2;
          a.l_out[orow] = L;
        }
        a.o_part_out[orow * D + d] = O;
      }
    } else {
      const int64_t prow = (int64_t)split * a.R + orow;
      if (d == 0) {
        a.ws_m[prow] = M * kLn2;
        a.ws_l[prow] = L;
      }
      a.ws_o[prow * D + d] = O;
    }
  }
  if (single || !a.merge_in_kernel) return;

  // ---- last CTA of the unit merges all splits (page: _merge_running, then O / l)
  __threadfence();
  ptx::named_bar_sync(1, kConsumerThreads);
  if (threadIdx.x == 0) {
    const unsigned prev = atomicAdd(a.counters + unit, 1u);
    flags[1] = (prev == (unsigned)(n_split_unit - 1)) ? 1 : 0;
  }
  ptx::named_bar_sync(1, kConsumerThreads);
  if (flags[1] == 0) return;
  __threadfence();
  for (int idx = threadIdx.x; idx < a.rows * D; idx += kConsumerThreads) {
    const int r = idx / D, d = idx - r * D;
    const int64_t orow = out_row(a, b, g_kv, r);
    float M = -CUDART_INF_F;
    for (int s2 = 0; s2 < n_split_unit; ++s2) M = fmaxf(M, __ldcg(a.ws_m + (int64_t)s2 * a.R + orow));
    float L = 0.f, O = 0.f;
    if (M != -CUDART_INF_F) {
      const float M2 = M * kLog2e;
      for (int s2 = 0; s2 < n_split_unit; ++s2) {
        const int64_t prow = (int64_t)s2 * a.R + orow;
        const float w = ptx::ex2(__ldcg(a.ws_m + prow) * kLog2e - M2);
        L += w * __ldcg(a.ws_l + prow);
        O += w * __ldcg(a.ws_o + prow * D + d);
      }
    }
    if (a.o != nullptr) {
      a.o[orow * D + d] = __float2half_rn(L > 0.f ? O / L : 0.f);
    } else {
      if (d == 0) {
        a.m_out[orow] = M;
        a.l_out[orow] = L;
      }
      a.o_part_out[orow * D + d] = O;
    }
  }
  if (threadIdx.x == 0) atomicExch(a.counters + unit, 0u);
}

// Public merge of n_parts partials laid out [n_parts][rows] and
// [n_parts][rows][D] (natural-log m).  One warp per row.
template <int D>
__global__ void __launch_bounds__(256)
gqa_merge_kernel(const float* __restrict__ m, const float* __restrict__ l, const float* __restrict__ op,
                 int n_parts, int64_t rows, __half* o, float* m_out, float* l_out, float* o_out) {
  constexpr int PER = D / 32;
  const int64_t r = (int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (r >= rows) return;
  float M = -CUDART_INF_F;
  for (int s = lane; s < n_parts; s += 32) M = fmaxf(M, m[(int64_t)s * rows + r]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
  float acc[PER];
#pragma unroll
  for (int i = 0; i < PER; ++i) acc[i] = 0.f;
  float L = 0.f;
  if (M != -CUDART_INF_F) {
    const float M2 = M * kLog2e;
    for (int s = 0; s < n_parts; ++s) {
      const int64_t pr = (int64_t)s * rows + r;
      const float w = ptx::ex2(m[pr] * kLog2e - M2);
      L += w * l[pr];
      const float* src = op + pr * D + lane * PER;
      if constexpr (PER == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] += w * v.x; acc[1] += w * v.y; acc[2] += w * v.z; acc[3] += w * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] += w * v.x; acc[1] += w * v.y;
      }
    }
  }
  if (o != nullptr) {
    const float inv = L > 0.f ? 1.f / L : 0.f;
#pragma unroll
    for (int i = 0; i < PER; ++i) o[r * D + lane * PER + i] = __float2half_rn(acc[i] * inv);
  } else {
    if (lane == 0) {
      m_out[r] = M;
      l_out[r] = L;
    }
#pragma unroll
    for (int i = 0; i < PER; ++i) o_out[r * D + lane * PER + i] = acc[i];
  }
}

}  // namespace gqa
