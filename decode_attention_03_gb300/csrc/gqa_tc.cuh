// Split-KV GQA decode on the 5th-generation tensor cores (tcgen05 + tensor memory), for
// units with many query rows: G*T_q up to 128 (speculative verification or the
// prefill-adjacent decode of several tokens per step).
//
// Same work decomposition as gqa_split_kernel (page "kernbench2 ...
// _gqa_attention_decode_long.py", "GQA fused-attention decode kernel -- long context":
// each split sweeps its key slice in tiles with a running (m, l, O); the unit's splits
// are folded with _merge_running), but the two products of a tile run as single-thread
// tcgen05.mma instructions with their accumulators in tensor memory instead of
// per-warp mma.sync fragments in registers, which cannot hold O for 128 rows:
//
//   S = Q K^T      M = 128 query rows (the unit's G*T_q rows, zero-padded), N = 64 keys,
//                  K = d_head; A = Q and B = the K tile, both K-major in shared memory
//                  with the 128-byte swizzle the TMA writes; S (fp32) in TMEM.
//   O += P V       M = 128 rows, N = d_head, K = 64 keys; A = P (f16 / bf16, written to
//                  shared memory by the softmax warps), B = the V tile read MN-major
//                  straight from its TMA layout; O (fp32) in TMEM.
//
// Warps: 0-7 softmax and epilogue in two warpgroups that take alternate tiles (thread =
// query row = TMEM lane, so a row's max and sum are thread-local; warpgroup wg owns S
// buffer wg, P buffer wg and its own O accumulator, and the two row states are combined
// in the epilogue), 8 the TMA producer, 9 and 10 the two MMA issuers: one thread issues
// S(t+2) as soon as the warpgroup has copied S(t) to registers, another issues PV(t) when
// P(t) is ready (a single issuer serialised the two chains: measured on GB300, tcgen05.mma
// and tcgen05.commit cost the issuing thread tens to hundreds of cycles each).
//
// Lazy rescaling: a row keeps the max it last rescaled to (m_used) and rescales its O only
// when a tile's max exceeds m_used by more than kTcRescale in log2 units (then p <=
// 2^kTcRescale fits the 16-bit P); a rescale never waits on the tensor core, because the
// warpgroup's previous PV has completed by the time its next S is ready.  The exact row
// max is tracked alongside and applied in the epilogue, so the emitted (m, l, O) equal
// the exact-max partial.
#pragma once
#include <cuda_runtime.h>

#include "gqa_kernels.cuh"

namespace gqa {

constexpr int kTcRows = 128;        // MMA M: query rows of a unit, zero-padded
constexpr int kTcKeys = 64;         // keys per tile (S MMA N, PV MMA K)
constexpr int kTcCols = 512;        // TMEM columns allocated: S buffers at [0, 64) and [64, 128),
constexpr int kTcOCol = 128;        //   O accumulators at [128, 128 + D) and [256, 256 + D)
constexpr int kTcOStride = 128;
constexpr float kTcRescale = 8.f;   // log2 growth of a row max that forces an O rescale
// tensor-memory columns: two S buffers below the first O accumulator, two O accumulators of up to
// 128 columns inside the allocation
static_assert(2 * kTcKeys <= kTcOCol && kTcOCol + kTcOStride + 128 <= kTcCols, "TMEM column map");

template <int D, int STAGES>
struct TcCfg {
  static constexpr int HALVES = D / 64;
  static constexpr int QPLANE = kTcRows * 128;           // [128 rows][64 columns], 128-byte swizzle
  static constexpr int KPLANE = kTcKeys * 128;           // [64 keys][64 columns]
  static constexpr int Q_BYTES = HALVES * QPLANE;
  static constexpr int P_BYTES = kTcRows * kTcKeys * 2;  // P of one tile: one [128 rows][64 keys] plane
  static constexpr int KV_BYTES = HALVES * KPLANE;       // one K (or V) tile
  static constexpr int STAGE_BYTES = 2 * KV_BYTES;
  static constexpr int Q_OFF = 0;
  static constexpr int P_OFF = Q_BYTES;
  static constexpr int RING_OFF = P_OFF + 2 * P_BYTES;
  static constexpr int CTRL_OFF = RING_OFF + STAGES * STAGE_BYTES;
  static constexpr int NBARS = 3 * STAGES + 7;
  static constexpr int CTRL_BYTES = NBARS * 8 + 16;
  static constexpr int SMEM_BYTES = 1024 + CTRL_OFF + CTRL_BYTES;
  static constexpr int SOFTMAX_THREADS = 8 * 32;   // two warpgroups
  static constexpr int TMA_WARP = 8;
  static constexpr int S_WARP = 9;                 // issues S = Q K^T
  static constexpr int PV_WARP = 10;               // issues O += P V; owns the TMEM allocation
  static constexpr int THREADS = 11 * 32;
};

// stages: as many 64-key K+V tiles as fit next to Q and the two P buffers, 3 to 8 (the
// warpgroups' wait on a stage barrier for their previous PV relies on at least 3)
template <int D>
constexpr int tc_stages() {
  constexpr int fixed = 1024 + TcCfg<D, 1>::RING_OFF + TcCfg<D, 8>::CTRL_BYTES;
  constexpr int n = (227 * 1024 - fixed) / TcCfg<D, 1>::STAGE_BYTES;
  return n > 8 ? 8 : n;
}

// pairwise (tree) reductions: log2(N) dependent steps instead of N - 1
template <int N>
__device__ __forceinline__ float tree_max(const float (&x)[N]) {
  float t[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; ++i) t[i] = fmaxf(x[i], x[i + N / 2]);
#pragma unroll
  for (int w = N / 4; w >= 1; w /= 2)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = fmaxf(t[i], t[i + w]);
  return t[0];
}

template <int N>
__device__ __forceinline__ float tree_min(const float (&x)[N]) {
  float t[N / 2];
#pragma unroll
  for (int i = 0; i < N / 2; ++i) t[i] = fminf(x[i], x[i + N / 2]);
#pragma unroll
  for (int w = N / 4; w >= 1; w /= 2)
#pragma unroll
    for (int i = 0; i < w; ++i) t[i] = fminf(t[i], t[i + w]);
  return t[0];
}

// Bounded wait for a phase by the whole warp; on give-up lane 0 records the timeout.
// Warp-uniform result.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, const DecodeArgs& a, volatile int* flags,
                                          int lane) {
  const bool ok = __all_sync(0xffffffffu, ptx::mbar_wait_bounded(ptx::smem_u32(bar), parity, a.timeout_ns, flags));
  if (!ok && lane == 0) raise_timeout(a, flags);
  return ok;
}

template <int D, int STAGES, bool CAUSAL, bool BF16>
__global__ void __launch_bounds__(TcCfg<D, STAGES>::THREADS, 1)
gqa_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
              const DecodeArgs a) {
  using C = TcCfg<D, STAGES>;
  static_assert(STAGES >= 3, "the previous-PV wait on a stage barrier needs three stages");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint64_t* k_full = reinterpret_cast<uint64_t*>(smem + C::CTRL_OFF);
  uint64_t* v_full = k_full + STAGES;
  uint64_t* empty = v_full + STAGES;       // PV of the stage's tile completed (commit): stage free,
                                           //   and that warpgroup's P buffer and O are free
  // per warpgroup wg (tiles t with t % 2 == wg): S buffer, P buffer and O accumulator wg
  uint64_t* s_full = empty + STAGES;       // [2] S(t) in TMEM (commit)
  uint64_t* s_empty = s_full + 2;          // [2] the warpgroup copied S(t) to registers (one arrival per active warp)
  uint64_t* p_full = s_full + 4;           // [2] P(t) in shared memory (one arrival per active warp)
  uint64_t* fin = s_full + 6;              // both issuers' MMAs completed (one commit each)
  volatile int* flags = reinterpret_cast<volatile int*>(k_full + C::NBARS);  // [0] abort [1] last [2] TMEM

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int g_kv = blockIdx.x, split = blockIdx.y, b = blockIdx.z;
  const int unit = b * a.h_kv + g_kv;
  const int nact = (a.rows + 31) >> 5;    // warps of a warpgroup holding real query rows
  const uint32_t sbase = ptx::smem_u32(smem);
  const Win ring{sbase + C::RING_OFF, sbase + C::CTRL_OFF, a.status};
  const Win qwin{sbase + C::Q_OFF, sbase + C::Q_OFF + C::Q_BYTES, a.status};
  const Win pwin{sbase + C::P_OFF, sbase + C::P_OFF + 2 * C::P_BYTES, a.status};

  const int64_t tiles_total = (a.s_len + kTile - 1) / kTile;
  const int64_t t0 = tiles_total * split / a.n_splits;
  const int64_t t1 = tiles_total * (split + 1) / a.n_splits;
  const int64_t key_begin = a.s_begin + t0 * kTile;
  const int64_t key_end = min(a.s_begin + t1 * kTile, a.s_begin + a.s_len);
  const int n_tiles = (int)(t1 - t0);

  if (threadIdx.x == 0) {
    for (int s = 0; s < STAGES; ++s) {
      ptx::mbar_init(ptx::smem_u32(k_full + s), 1);
      ptx::mbar_init(ptx::smem_u32(v_full + s), 1);
      ptx::mbar_init(ptx::smem_u32(empty + s), 1);
    }
    for (int i = 0; i < 2; ++i) {
      ptx::mbar_init(ptx::smem_u32(s_full + i), 1);
      ptx::mbar_init(ptx::smem_u32(s_empty + i), nact);
      ptx::mbar_init(ptx::smem_u32(p_full + i), nact);
    }
    ptx::mbar_init(ptx::smem_u32(fin), 2);
    flags[0] = 0;
    flags[1] = 0;
    ptx::fence_mbar_init();
  }
  if (warp == C::PV_WARP) {
    ptx::tmem_alloc(ptx::smem_u32((const void*)(flags + 2)), kTcCols);
    ptx::tmem_relinquish();
  }
  if (warp == C::TMA_WARP && lane == 0) {
    ptx::prefetch_tensormap(&tmK);
    ptx::prefetch_tensormap(&tmV);
  }
  ptx::tc_fence_before();
  __syncthreads();
  ptx::tc_fence_after();
  const uint32_t tmem = (uint32_t)flags[2];
  // the first ring's worth of K and V boxes into L2 while the previous kernel in the stream may
  // still run (a hint: the loads after the dependency wait read whatever it wrote)
  if (warp == C::TMA_WARP && lane == 0) {
    for (int it = 0; it < n_tiles && it < STAGES; ++it) {
      const int64_t y = (int64_t)b * a.S_kv + key_begin + (int64_t)it * kTcKeys;
      if (y < (int64_t)a.B * a.S_kv && g_kv < a.h_kv) {
        ptx::tma_prefetch_3d(&tmK, 0, (int)y, g_kv * C::HALVES);
        ptx::tma_prefetch_3d(&tmV, 0, (int)y, g_kv * C::HALVES);
      }
    }
  }
  // launched as a programmatic dependent: the set-up above (barriers, tensor memory) may overlap the
  // previous kernel in the stream; nothing in global memory is touched before it has completed
  ptx::grid_dependency_wait();

  if (warp == C::TMA_WARP) {
    // ------------------------------------------------------------ TMA producer
    if (lane == 0) {
      const uint64_t pol = ptx::policy_evict_first();
      const int stall_tile = (a.stall_cta >= 0 &&
                              a.stall_cta == (int)(blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z)))
                                 ? 1 : -1;
      const int64_t y_base = (int64_t)b * a.S_kv;
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
        const uint32_t kdst = ptx::smem_u32(smem + C::RING_OFF + s * C::STAGE_BYTES);
        const int64_t y = y_base + key_begin + (int64_t)it * kTcKeys;
        // the boxes start inside K / V's rows and heads and land inside the ring (else the stage
        // completes without data: the check has recorded it)
        if (idx_ok(y, (int64_t)a.B * a.S_kv, a.status) && idx_ok(g_kv, a.h_kv, a.status) &&
            smem_ok(kdst, C::STAGE_BYTES, ring.lo, ring.hi, a.status)) {
          ptx::mbar_arrive_expect_tx(ptx::smem_u32(k_full + s), C::KV_BYTES);
          ptx::tma_load_3d(kdst, &tmK, ptx::smem_u32(k_full + s), 0, (int)y, g_kv * C::HALVES, pol);
          ptx::mbar_arrive_expect_tx(ptx::smem_u32(v_full + s), C::KV_BYTES);
          ptx::tma_load_3d(kdst + C::KV_BYTES, &tmV, ptx::smem_u32(v_full + s), 0, (int)y, g_kv * C::HALVES, pol);
        } else {
          ptx::mbar_arrive(ptx::smem_u32(k_full + s));
          ptx::mbar_arrive(ptx::smem_u32(v_full + s));
        }
      }
      if (gave_up || stall_tile >= 0) {
        // wait (bounded) for copies still in flight before the CTA can exit
        for (int it = max(0, issued - STAGES); it < issued; ++it) {
          if (it == stall_tile) continue;
          const uint32_t ph = (uint32_t)(it / STAGES) & 1u;
          ptx::mbar_wait_bounded(ptx::smem_u32(k_full + (it % STAGES)), ph, a.timeout_ns, nullptr);
          ptx::mbar_wait_bounded(ptx::smem_u32(v_full + (it % STAGES)), ph, a.timeout_ns, nullptr);
        }
      }
    }
  } else if (warp == C::S_WARP) {
    // ------------------------------------------------------------ S issuer: S(t) = Q K(t)^T
    constexpr uint32_t kIdS = ptx::idesc_f16(kTcRows, kTcKeys, BF16, false, false);
    // descriptors of k-step 0; k-step kk adds its byte offset / 16 to the start-address field
    const uint64_t dq = ptx::smem_desc_sw128(ptx::smem_u32(smem + C::Q_OFF), 16, 1024);
    const uint64_t dk = ptx::smem_desc_sw128(ptx::smem_u32(smem + C::RING_OFF), 16, 1024);
    ptx::named_bar_sync(2, 4 * 32 + 32);   // Q is in shared memory (written by warpgroup 0)
    for (int it = 0; it < n_tiles; ++it) {
      const int s = it % STAGES;
      if (!warp_wait(k_full + s, (uint32_t)(it / STAGES) & 1u, a, flags, lane)) break;
      // S buffer it % 2 was copied out by its warpgroup (tile it - 2)
      if (it >= 2 && !warp_wait(s_empty + (it & 1), (uint32_t)((it >> 1) - 1) & 1u, a, flags, lane)) break;
      ptx::tc_fence_after();
      if (lane == 0) {
        const uint64_t dks = dk + (uint64_t)((s * C::STAGE_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off_q = (kk >> 2) * C::QPLANE + (kk & 3) * 32;
          const uint32_t off_k = (kk >> 2) * C::KPLANE + (kk & 3) * 32;
          ptx::tc_mma_ss(tmem + (it & 1) * kTcKeys, dq + (off_q >> 4), dks + (off_k >> 4), kIdS, kk > 0 ? 1u : 0u);
        }
        ptx::tc_commit(ptx::smem_u32(s_full + (it & 1)));
      }
      __syncwarp();
    }
    if (lane == 0) ptx::tc_commit(ptx::smem_u32(fin));
    __syncwarp();
  } else if (warp == C::PV_WARP) {
    // ------------------------------------------------------------ PV issuer: O(t % 2) += P(t) V(t)
    constexpr uint32_t kIdPV = ptx::idesc_f16(kTcRows, D, BF16, false, true);
    const uint64_t dp = ptx::smem_desc_sw128(ptx::smem_u32(smem + C::P_OFF), 16, 1024);
    // V as the MN-major B operand: 64-column planes KPLANE bytes apart (leading), 8-key groups
    // 1024 bytes apart (stride)
    const uint64_t dv = ptx::smem_desc_sw128(ptx::smem_u32(smem + C::RING_OFF + C::KV_BYTES), C::KPLANE, 1024);
    for (int t = 0; t < n_tiles; ++t) {
      const int s = t % STAGES;
      if (!warp_wait(v_full + s, (uint32_t)(t / STAGES) & 1u, a, flags, lane)) break;
      if (!warp_wait(p_full + (t & 1), (uint32_t)(t >> 1) & 1u, a, flags, lane)) break;
      if (t == n_tiles - 1) {
        // keys past the slice: zero their V rows so that 0 * (anything) cannot reach O
        const int valid = (int)(key_end - (key_begin + (int64_t)t * kTcKeys));
        uint8_t* vrow = smem + C::RING_OFF + s * C::STAGE_BYTES + C::KV_BYTES;
        for (int i = lane; i < (kTcKeys - valid) * 8 * C::HALVES; i += 32) {
          const int row = valid + i / (8 * C::HALVES), rem = i % (8 * C::HALVES);
          uint8_t* dst = vrow + (rem >> 3) * C::KPLANE + row * 128 + (rem & 7) * 16;
          if (smem_ok(ptx::smem_u32(dst), 16, ring.lo, ring.hi, a.status))
            *reinterpret_cast<uint4*>(dst) = make_uint4(0u, 0u, 0u, 0u);
        }
        ptx::fence_proxy_async_smem();
        __syncwarp();
      }
      ptx::tc_fence_after();
      if (lane == 0) {
        const uint64_t dps = dp + (uint64_t)(((t & 1) * C::P_BYTES) >> 4);
        const uint64_t dvs = dv + (uint64_t)((s * C::STAGE_BYTES) >> 4);
#pragma unroll
        for (int kk = 0; kk < kTcKeys / 16; ++kk)
          // the first PV of each accumulator overwrites it
          ptx::tc_mma_ss(tmem + kTcOCol + (t & 1) * kTcOStride, dps + (uint64_t)((kk * 32) >> 4),
                         dvs + (uint64_t)((kk * 16 * 128) >> 4), kIdPV, (t >= 2 || kk > 0) ? 1u : 0u);
        ptx::tc_commit(ptx::smem_u32(empty + s));
      }
      __syncwarp();
    }
    // both issuers' MMAs complete before the tensor memory is released
    if (lane == 0) {
      ptx::tc_commit(ptx::smem_u32(fin));
      ptx::mbar_wait_bounded(ptx::smem_u32(fin), 0u, a.timeout_ns, nullptr);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax / epilogue warpgroups
    const int wg = warp >> 2;                             // tiles t with t % 2 == wg
    const int r = (warp & 3) * 32 + lane;                 // query row = TMEM lane
    const uint32_t t_lane = (uint32_t)((warp & 3) * 32) << 16;
    const uint32_t tmem_s = tmem + t_lane + wg * kTcKeys;
    const uint32_t tmem_o = tmem + t_lane + kTcOCol + wg * kTcOStride;
    if (wg == 0) {
      // Q row r into HALVES swizzled [128][64] planes; rows past the unit are zero
      uint8_t* qs = smem + C::Q_OFF;
      const uint4* src = r < a.rows && idx_ok(out_row(a, b, g_kv, r), a.R, a.status)
                             ? reinterpret_cast<const uint4*>(a.q + out_row(a, b, g_kv, r) * D)
                             : nullptr;
#pragma unroll
      for (int c = 0; c < D / 8; ++c) {
        const uint4 v = src ? __ldg(src + c) : make_uint4(0u, 0u, 0u, 0u);
        uint8_t* dst = qs + (c >> 3) * C::QPLANE + r * 128 + (((c & 7) ^ (r & 7)) << 4);
        if (smem_ok(ptx::smem_u32(dst), 16, qwin.lo, qwin.hi, a.status)) *reinterpret_cast<uint4*>(dst) = v;
      }
      ptx::fence_proxy_async_smem();
      ptx::named_bar_arrive(2, 4 * 32 + 32);
    }
    const float c2 = a.scale_log2;
    const int64_t lim = CAUSAL ? a.S_kv - a.T_q + r / a.G : INT64_MAX;   // last key this row may see
    float m_used = -CUDART_INF_F;   // reference max of l and O (log2 domain of scaled logits)
    float m_seen = -CUDART_INF_F;   // exact running max
    float l = 0.f;
    uint8_t* prow = smem + C::P_OFF + wg * C::P_BYTES + r * 128;
    if ((warp & 3) < nact) {
      for (int it = wg; it < n_tiles; it += 2) {
        if (!warp_wait(s_full + wg, (uint32_t)(it >> 1) & 1u, a, flags, lane)) break;
        ptx::tc_fence_after();
        float x[kTcKeys];   // raw scores q.k of this row against the tile's keys
        {
          static_assert(kTcKeys == 64, "one 64-column load per tile");
          uint32_t u[64];
          ptx::tmem_ld64(tmem_s, u);
#pragma unroll
          for (int j = 0; j < 64; ++j) x[j] = __uint_as_float(u[j]);
        }
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(s_empty + wg));   // S(it + 2) may overwrite it

        const int64_t key0 = key_begin + (int64_t)it * kTcKeys;
        int64_t vis = key_end - key0;                          // keys of the tile this row sees
        if (CAUSAL) vis = min(vis, lim - key0 + 1);
        const bool whole = vis >= kTcKeys;
        // tile max of the scaled logits (log2 domain); -inf when the row sees no key
        float mt;
        if (whole) {
          mt = (c2 >= 0.f ? tree_max(x) : tree_min(x)) * c2;   // the scale folds into the exponent below
        } else {
#pragma unroll
          for (int j = 0; j < kTcKeys; ++j) x[j] = j < vis ? x[j] * c2 : -CUDART_INF_F;
          mt = tree_max(x);
        }
        m_seen = fmaxf(m_seen, mt);
        // PV(it - 2) -- the previous use of this warpgroup's P buffer and O -- must be complete
        // before O is rescaled or P rewritten; it signals the stage barrier of tile it - 2
        bool prev_done = it < 2;
        const int tp = it - 2;
        const bool need = mt > m_used + kTcRescale;
        if (__any_sync(0xffffffffu, need)) {
          const float m_new = need ? mt : m_used;
          const float alpha = need ? ptx::ex2(m_used - m_new) : 1.f;   // m_used = -inf -> 0
          l *= alpha;
          m_used = m_new;
          if (it >= 2) {
            if (!warp_wait(empty + tp % STAGES, (uint32_t)(tp / STAGES) & 1u, a, flags, lane)) break;
            prev_done = true;
            ptx::tc_fence_after();
#pragma unroll
            for (int c = 0; c < D / 32; ++c) {
              uint32_t u[32];
              ptx::tmem_ld32(tmem_o + c * 32, u);
#pragma unroll
              for (int j = 0; j < 32; ++j) u[j] = __float_as_uint(__uint_as_float(u[j]) * alpha);
              ptx::tmem_st32(tmem_o + c * 32, u);
            }
            ptx::tmem_wait_st();
          }
        }
        const float mu = m_used == -CUDART_INF_F ? 0.f : m_used;
        uint32_t pk[kTcKeys / 2];
        float lp[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) lp[i] = 0.f;
        if (whole) {
          const float nmu = -mu;
#pragma unroll
          for (int j = 0; j < kTcKeys; j += 2) {
            const float p0 = ptx::ex2(fmaf(x[j], c2, nmu)), p1 = ptx::ex2(fmaf(x[j + 1], c2, nmu));
            lp[(j / 2) & 7] += p0 + p1;
            pk[j / 2] = Elem<BF16>::pack(p0, p1);
          }
        } else {
#pragma unroll
          for (int j = 0; j < kTcKeys; j += 2) {
            const float p0 = ptx::ex2(x[j] - mu), p1 = ptx::ex2(x[j + 1] - mu);
            lp[(j / 2) & 7] += p0 + p1;
            pk[j / 2] = Elem<BF16>::pack(p0, p1);
          }
        }
        l += ((lp[0] + lp[1]) + (lp[2] + lp[3])) + ((lp[4] + lp[5]) + (lp[6] + lp[7]));
        if (!prev_done && !warp_wait(empty + tp % STAGES, (uint32_t)(tp / STAGES) & 1u, a, flags, lane)) break;
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          uint8_t* dst = prow + ((c ^ (r & 7)) << 4);
          if (smem_ok(ptx::smem_u32(dst), 16, pwin.lo, pwin.hi, a.status))
            *reinterpret_cast<uint4*>(dst) = make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        ptx::fence_proxy_async_smem();
        ptx::tc_fence_before();
        __syncwarp();
        if (lane == 0) ptx::mbar_arrive(ptx::smem_u32(p_full + wg));
      }
    }

    // ------------------------------------------------------------ epilogue
    if (threadIdx.x == 0) ptx::grid_launch_dependents();   // a separate merge kernel may start launching
    // a wait that gave up anywhere -> leave the output alone
    const bool aborted = ptx::named_bar_or(1, C::SOFTMAX_THREADS, flags[0] != 0);
    const int n_mine = n_tiles > wg ? (n_tiles - wg + 1) / 2 : 0;   // tiles of this warpgroup
    bool ready = !aborted;
    if (ready && (warp & 3) < nact && n_mine > 0) {
      const int t = wg + 2 * (n_mine - 1);                          // its last tile
      ready = warp_wait(empty + t % STAGES, (uint32_t)(t / STAGES) & 1u, a, flags, lane);
      ptx::tc_fence_after();
    }
    // every PV has completed past this barrier (or something gave up)
    const bool stop = ptx::named_bar_or(1, C::SOFTMAX_THREADS, !ready);
    if (!stop) {
      // warpgroup 1 hands its row state to warpgroup 0 through its (now idle) P buffer
      float* xchg = reinterpret_cast<float*>(smem + C::P_OFF + C::P_BYTES);
      if (wg == 1) {
        xchg[r] = m_used;
        xchg[kTcRows + r] = m_seen;
        xchg[2 * kTcRows + r] = l;
      }
      ptx::named_bar_sync(1, C::SOFTMAX_THREADS);
      const bool single = (a.n_splits == 1);
      if (wg == 0 && (warp & 3) < nact) {
        // combine the two warpgroups' partials of row r (exact max M, each side rescaled to it)
        const float mu1 = xchg[r], ms1 = xchg[kTcRows + r], l1 = xchg[2 * kTcRows + r];
        const float M = fmaxf(m_seen, ms1);
        const float f0 = m_used == -CUDART_INF_F ? 0.f : ptx::ex2(m_used - M);
        const float f1 = mu1 == -CUDART_INF_F ? 0.f : ptx::ex2(mu1 - M);
        const float L = l * f0 + l1 * f1;
        const bool has0 = n_tiles > 0, has1 = n_tiles > 1;
        // a real row, whose output (or partial) row and split slot are in range
        const bool row_ok = r < a.rows && idx_ok(out_row(a, b, g_kv, r), a.R, a.status) &&
                            (single || idx_ok(split, a.n_splits, a.status));
        const int64_t orow = out_row(a, b, g_kv, row_ok ? r : 0);
        const float inv = L > 0.f ? 1.f / L : 0.f;
        const uint32_t o0 = tmem + t_lane + kTcOCol, o1 = o0 + kTcOStride;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t u0[32], u1[32];
          if (has0) {
            ptx::tmem_ld32(o0 + c * 32, u0);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) u0[j] = 0u;
          }
          if (has1) {
            ptx::tmem_ld32(o1 + c * 32, u1);
          } else {
#pragma unroll
            for (int j = 0; j < 32; ++j) u1[j] = 0u;
          }
          float ov[32];
#pragma unroll
          for (int j = 0; j < 32; ++j) ov[j] = __uint_as_float(u0[j]) * f0 + __uint_as_float(u1[j]) * f1;
          if (!row_ok) continue;
          if (single && a.o != nullptr) {
            uint4* dst = reinterpret_cast<uint4*>(a.o + orow * D + c * 32);
#pragma unroll
            for (int q4 = 0; q4 < 4; ++q4) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e)
                w[e] = Elem<BF16>::pack(ov[q4 * 8 + 2 * e] * inv, ov[q4 * 8 + 2 * e + 1] * inv);
              dst[q4] = make_uint4(w[0], w[1], w[2], w[3]);
            }
          } else {
            float* op = single ? a.o_part_out + orow * D : a.ws_o + ((int64_t)split * a.R + orow) * D;
            float4* dst = reinterpret_cast<float4*>(op + c * 32);
#pragma unroll
            for (int q4 = 0; q4 < 8; ++q4)
              dst[q4] = make_float4(ov[4 * q4], ov[4 * q4 + 1], ov[4 * q4 + 2], ov[4 * q4 + 3]);
          }
        }
        if (row_ok && !(single && a.o != nullptr)) {
          const float mn = M * kLn2;
          if (single) {
            a.m_out[orow] = mn;
            a.l_out[orow] = L;
          } else {
            a.ws_m[(int64_t)split * a.R + orow] = mn;
            a.ws_l[(int64_t)split * a.R + orow] = L;
          }
        }
      }
      // the last CTA of the unit folds the splits
      if (!single && a.merge_in_kernel && last_to_arrive<C::SOFTMAX_THREADS>(a, unit, a.n_splits, flags)) {
        const int n_items = a.rows * (D / 4);
        for (int i0 = 0; i0 < n_items; i0 += C::SOFTMAX_THREADS * 2)
          merge_pass<D, C::SOFTMAX_THREADS, 2, BF16>(a, b, g_kv, i0, a.n_splits);
        if (threadIdx.x == 0 && idx_ok(unit, (int64_t)a.B * a.h_kv, a.status)) atomicExch(a.counters + unit, 0u);
      }
    }
  }

  // release the tensor memory once every warp is done with it
  __syncwarp();
  ptx::tc_fence_before();
  __syncthreads();
  if (warp == C::PV_WARP) {
    ptx::tc_fence_after();
    ptx::tmem_dealloc(tmem, kTcCols);
  }
}

template <int D, bool CAUSAL, bool BF16>
struct TcInst {
  static constexpr int STAGES = tc_stages<D>();
  using C = TcCfg<D, STAGES>;
  static_assert(C::SMEM_BYTES <= 227 * 1024, "shared memory budget");

  static cudaError_t prepare(int* occupancy) {
    auto fn = gqa_tc_kernel<D, STAGES, CAUSAL, BF16>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, C::SMEM_BYTES);
    if (e != cudaSuccess) return e;
    return cudaOccupancyMaxActiveBlocksPerMultiprocessor(occupancy, fn, C::THREADS, C::SMEM_BYTES);
  }
  static cudaError_t launch(dim3 grid, cudaStream_t st, const CUtensorMap& tk, const CUtensorMap& tv,
                            const DecodeArgs& a) {
    return launch_dependent(gqa_tc_kernel<D, STAGES, CAUSAL, BF16>, grid, C::THREADS, C::SMEM_BYTES, st,
                            dim3(1, 1, 1), tk, tv, a);
  }
};

// One translation unit per d_head: variants (causal, bf16).
#define GQA_TC_CASES(D, CALL)                                                                    \
  if (!bf16) return causal ? TcInst<D, true, false>::CALL : TcInst<D, false, false>::CALL;       \
  return causal ? TcInst<D, true, true>::CALL : TcInst<D, false, true>::CALL;

#define GQA_DEFINE_TC_UNIT(NAME, D)                                                              \
  cudaError_t NAME##_prepare(int causal, int bf16, int* occupancy) {                             \
    GQA_TC_CASES(D, prepare(occupancy))                                                          \
  }                                                                                              \
  cudaError_t NAME##_launch(int causal, int bf16, dim3 grid, cudaStream_t st, const CUtensorMap& tk, \
                            const CUtensorMap& tv, const DecodeArgs& a) {                        \
    GQA_TC_CASES(D, launch(grid, st, tk, tv, a))                                                 \
  }

#define GQA_DECLARE_TC_UNIT(NAME)                                                                \
  cudaError_t NAME##_prepare(int causal, int bf16, int* occupancy);                              \
  cudaError_t NAME##_launch(int causal, int bf16, dim3 grid, cudaStream_t st, const CUtensorMap& tk, \
                            const CUtensorMap& tv, const DecodeArgs& a);

GQA_DECLARE_TC_UNIT(tc_d64)
GQA_DECLARE_TC_UNIT(tc_d128)

}  // namespace gqa
