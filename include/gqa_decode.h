/*
 * gqa_decode.h -- C ABI of the GB300 (sm_103a) GQA split-KV decode attention library
 * (libgqa_decode.so).
 *
 * The operation (page "kernbench2 ... _gqa_attention_decode_long.py", "GQA
 * fused-attention decode kernel -- long context": kernel docstring "Tensor
 * layout", the local tile math and "Final normalise + store"): for every
 * sequence b, query token t < T_q and query head h < h_q, with G = h_q / h_kv
 * query heads sharing KV head g = h / G,
 *
 *     O[b,t,h,:] = softmax_j( scale * Q[b,t,h,:] . K[b,j,g,:] ) . V[b,j,g,:]
 *
 * The key axis is swept in tiles and splits; every split yields a partial
 * (m, l, O) -- m the row max of the scaled logits (natural-log units), l the sum
 * of exp(logit - m), O the unnormalised sum of exp(logit - m) * V -- and partials
 * are folded with the page's online-softmax merge (_merge_running):
 * m = max(m_a, m_b), each side rescaled by exp(m_side - m), l and O summed.
 * The paged variant is page "muh_kernel_map.py", VLLM_KERNEL_MAP
 * 'paged_attention_v2': a per-partition pass plus a cross-partition merge.
 *
 * Conventions for every call
 *  - 16-bit buffers hold IEEE binary16 values (or bfloat16 with gqa_options.bf16), passed as
 *    uint16_t; float buffers are fp32.
 *  - All tensors are dense row-major, in device memory of the CURRENT CUDA
 *    device, 16-byte aligned.  The caller owns every buffer; the library never
 *    allocates device memory and never synchronises (except gqa_workspace_check).
 *  - `stream` is a cudaStream_t (NULL = legacy default stream).  Calls are
 *    asynchronous; arguments are validated on the host before any launch and
 *    a failed validation returns an error code without touching the GPU.
 *  - Launch failures return GQA_ERR_CUDA.  Faults detected on the device (a
 *    bounded wait that gave up, a block id outside the pool) are recorded in
 *    the workspace's status word; gqa_workspace_check reads it.
 *  - Supported: h_q % h_kv == 0, d_head in {64, 128}, G * T_q <= 128 for contiguous calls
 *    and G <= 64 for paged calls (GQA_ERR_UNSUPPORTED otherwise); no C++ exception crosses
 *    this ABI.
 *  - Two tensor-core paths compute the same result: the warp-level mma.sync split kernel
 *    (G * T_q <= 64) and the tcgen05 kernel (single-thread MMAs with fp32 accumulators in
 *    tensor memory, M = 128 query rows; contiguous calls, G * T_q <= 128), chosen by
 *    gqa_options.mma_path.
 *  - Scores, softmax statistics, partials and accumulation are fp32; the output
 *    O is rounded to f16 (nearest even).
 */
#ifndef GQA_DECODE_H_
#define GQA_DECODE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  GQA_OK = 0,
  GQA_ERR_INVALID_ARG = 1, /* null/misaligned pointer, bad size or range, bad block id (device) */
  GQA_ERR_UNSUPPORTED = 2, /* d_head or G*T_q outside the supported set */
  GQA_ERR_WORKSPACE = 3,   /* workspace smaller than the size query asks for */
  GQA_ERR_CUDA = 4,        /* a CUDA runtime/driver call or a launch failed */
  GQA_ERR_TIMEOUT = 5,     /* a bounded device wait gave up (reported by gqa_workspace_check) */
  GQA_ERR_BOUNDS = 6       /* checked build only: a device bounds check failed (gqa_workspace_check) */
} gqa_status;

/* Bits of gqa_build_flags(). */
#define GQA_BUILD_BOUNDS_CHECK 1 /* every computed global- and shared-memory offset of the kernels is
                                    range-checked on the device; a failure sets a status bit
                                    (GQA_ERR_BOUNDS) and skips the access -- nothing traps */

/* Optional knobs for tests and benchmarks (NULL = defaults everywhere). */
typedef struct {
  int n_splits;          /* contiguous calls: splits per (sequence, KV head); 0 = automatic: about
                            1.25 CTAs per SM, or, where the (sequence, KV head) units divide the
                            SM count into more than 16 splits of at least 48 64-key tiles (d_head
                            128, up to 8 rows, no causal tail), one CTA per SM running a deeper
                            ring; a forced count keeps the plain kernel */
  int merge_mode;        /* how a unit's splits are folded.  0 = automatic: on the mma.sync kernel
                            a cluster (3) for 2 to 16 splits where the cluster variant keeps the
                            plain kernel's ring depth (not at d_head 128 with more than 32 rows)
                            and the GPU holds every unit's cluster at once (one wave; the
                            runtime's count of co-resident clusters of that size), and one
                            cluster of 16 where the heuristic wants more than 16 splits over at
                            most 16 x 8 tiles (short sweeps);
                            otherwise, and always after the tcgen05 kernel, the separate merge
                            kernel.  1 = separate merge kernel.  2 = the last-arriving CTA of the
                            unit folds the splits in the same kernel (only on request).  3 = the
                            unit's splits (at most 16; more are capped) run as one thread-block
                            cluster and fold their partials through distributed shared memory, no
                            workspace partials and one launch (mma.sync kernel only: the automatic
                            mma_path takes it for up to 64 rows; GQA_ERR_UNSUPPORTED on the tcgen05
                            kernel) */
  uint32_t timeout_us;   /* limit of every device wait; 0 = 1,000,000 us */
  int test_stall_cta;    /* test hook, -1 = off.  Contiguous calls: linear id (x + X*(y + Y*z)) of
                            one CTA whose producer never loads its second tile; paged calls: the
                            index of one work item (partition x head group, in queue order) whose
                            second tile is never loaded.  The waits on that tile run out; use with
                            a small timeout_us.  The call then reports GQA_ERR_TIMEOUT through
                            gqa_workspace_check and the workspace must be re-initialised. */
  int paged_head_group;  /* paged calls: KV heads per work item and per TMA box, 1, 2 or 4 (must divide
                            h_kv; 2 and 4 need h_q / h_kv <= 16); 0 = 4, 2 or 1, the largest that fits */
  int causal;            /* contiguous calls with T_q > 1 (speculative verification): query token t
                            sees only the keys j <= S_kv - T_q + t (the T_q new tokens are the last
                            T_q keys); 0 = every token sees all S_kv keys.  No counterpart on the
                            pages (their kernel is stated for T_q = 1). */
  int bf16;              /* decode, partial and paged calls: q, k, v (and o) hold bfloat16 values
                            instead of IEEE binary16; arithmetic stays fp32, o is rounded to bf16 */
  int mma_path;          /* contiguous calls: 0 = automatic (tcgen05 when G * T_q >= 16, else mma.sync),
                            1 = mma.sync split kernel (G * T_q <= 64), 2 = tcgen05 kernel
                            (G * T_q <= 128).  The workspace size query covers either path. */
} gqa_options;

/* Default options: n_splits 0, merge_mode 0, timeout_us 0, test_stall_cta -1, paged_head_group 0,
 * causal 0, bf16 0, mma_path 0. */
gqa_options gqa_default_options(void);

/* Static text for a status code. */
const char* gqa_status_string(int status);

/* Library version, major*10000 + minor*100 + patch. */
int gqa_version(void);

/* How this library was built: GQA_BUILD_BOUNDS_CHECK for the checked build (libgqa_decode_checked.so,
 * compiled with GQA_BOUNDS_CHECK=1; slower, for tests and debugging), 0 for the regular one. */
int gqa_build_flags(void);

/* Splits per (sequence, KV head) the automatic plan picks on the current device for a contiguous
 * call with default options sweeping S_kv keys (gqa_options.n_splits); <= 0 on invalid arguments
 * or when no device is usable. */
int gqa_decode_num_splits(int batch, int T_q, int64_t S_kv, int h_q, int h_kv, int d_head);

/* What a gqa_decode_ex call with these shapes and options (NULL = defaults) launches on the current
 * device: splits per (sequence, KV head), the MMA path (1 mma.sync, 2 tcgen05) and the number of
 * kernel launches (1, or 2 with the separate merge kernel).  Output pointers may be NULL. */
gqa_status gqa_decode_plan(int batch, int T_q, int64_t S_kv, int h_q, int h_kv, int d_head, const gqa_options* opt,
                           int* n_splits, int* mma_path, int* launches);

/* Decode kernel of a contiguous call (gqa_decode_plan_ex). */
#define GQA_KERNEL_SPLIT 0         /* mma.sync split kernel, about 1.25 CTAs per SM */
#define GQA_KERNEL_SPLIT_CLUSTER 1 /* its cluster variant: a unit's splits are the CTAs of one cluster */
#define GQA_KERNEL_SPLIT_DEEP 2    /* its deep-ring variant: one CTA per SM, a deeper TMA ring */
#define GQA_KERNEL_TCGEN05 3       /* tcgen05 kernel, accumulators in tensor memory */
/* How the splits of a unit are folded (gqa_decode_plan_ex). */
#define GQA_FOLD_NONE 0            /* one split: the kernel normalises and writes the output */
#define GQA_FOLD_CLUSTER 1         /* in the cluster, through distributed shared memory */
#define GQA_FOLD_MERGE_KERNEL 2    /* by the merge kernel, launched as a programmatic dependent */
#define GQA_FOLD_LAST_CTA 3        /* by the unit's last-arriving CTA (merge_mode 2) */

/* gqa_decode_plan, and which kernel runs (GQA_KERNEL_*) and how its splits are folded (GQA_FOLD_*).
 * No counterpart on the pages: a query of this library's own plan.  Output pointers may be NULL. */
gqa_status gqa_decode_plan_ex(int batch, int T_q, int64_t S_kv, int h_q, int h_kv, int d_head,
                              const gqa_options* opt, int* n_splits, int* mma_path, int* launches, int* kernel,
                              int* fold);

/* Workspace bytes for gqa_decode / gqa_decode_partial on the current device, sweeping S_kv
 * keys (for a partial call pass s_len).  n_splits = 0 sizes for the heuristic; a positive
 * value sizes for that forced split count.  Returns 0 on invalid arguments.  The workspace
 * holds a status word, one arrival counter per (sequence, KV head) and the split partials. */
size_t gqa_decode_workspace_size(int batch, int T_q, int64_t S_kv, int h_q, int h_kv, int d_head,
                                 int n_splits);

/* Workspace bytes for a gqa_decode call with the automatic split count on the current device:
 * gqa_decode_workspace_size(batch, T_q, S_kv, h_q, h_kv, d_head, 0).  0 on invalid arguments or
 * when no device is usable. */
size_t gqa_workspace_size(int batch, int T_q, int64_t S_kv, int h_q, int h_kv, int d_head);

/* Workspace bytes for gqa_decode_paged and gqa_decode_paged_vllm (T_q = 1); partition_size 0 sizes
 * for the automatic choice.  Returns 0 on invalid arguments. */
size_t gqa_paged_workspace_size(int num_seqs, int h_q, int h_kv, int d_head, int max_seq_len,
                                int partition_size);

/* What a paged call (vllm_layout 0: gqa_decode_paged, 1: gqa_decode_paged_vllm) with these shapes
 * and options (NULL = defaults) does on the current device: the partition size (the automatic
 * choice resolved), the KV heads per work item, and the kernel launches (two per 1024 sequences
 * when some sequence spans several partitions, else one).  Outputs may be NULL. */
gqa_status gqa_paged_plan(int num_seqs, int h_q, int h_kv, int d_head, int block_size, int max_seq_len,
                          int partition_size, int vllm_layout, const gqa_options* opt, int* partition_out,
                          int* head_group_out, int* launches_out);

/* Zero-fill a workspace (asynchronous memset on `stream`).  A workspace must be zero before
 * its first use; every call that completes without a device fault leaves it so again. */
gqa_status gqa_workspace_init(void* workspace, size_t ws_bytes, void* stream);

/* Synchronise `stream`, read and clear the workspace's device status word.  Returns GQA_OK,
 * GQA_ERR_TIMEOUT (a bounded wait gave up; outputs of that call are invalid and the
 * workspace must be re-initialised), GQA_ERR_INVALID_ARG (a block id or sequence length
 * outside the pool / table was seen; affected outputs are invalid) or, in the checked build
 * only, GQA_ERR_BOUNDS (a device bounds check failed: a library fault; outputs invalid). */
gqa_status gqa_workspace_check(void* workspace, void* stream);

/* Full decode step (contiguous KV).
 *   q  (batch, T_q, h_q*d_head) f16      k, v (batch, S_kv, h_kv*d_head) f16
 *   o  (batch, T_q, h_q*d_head) f16, written
 * Every query token attends to all S_kv >= 1 keys of its sequence (no causal mask).
 * `scale` multiplies q.k (e.g. 1/sqrt(d_head)).  batch = 0 is a no-op.
 * batch * S_kv must be < 2^31. */
gqa_status gqa_decode(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o,
                      int batch, int T_q, int64_t S_kv, int h_q, int h_kv, int d_head, float scale,
                      void* workspace, size_t ws_bytes, void* stream);

gqa_status gqa_decode_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o,
                         int batch, int T_q, int64_t S_kv, int h_q, int h_kv, int d_head, float scale,
                         void* workspace, size_t ws_bytes, void* stream, const gqa_options* opt);

/* Partial over keys [s_begin, s_begin + s_len) of every sequence (0 <= s_begin,
 * s_begin + s_len <= S_kv; s_len = 0 gives the empty partial m = -inf, l = 0, O = 0, and then
 * k and v are not read and may be NULL, with S_kv = 0 for a caller that holds no keys).
 * Outputs, rows ordered like Q's (b, t, h): m, l (batch*T_q*h_q) fp32 and the
 * unnormalised o_part (batch*T_q*h_q, d_head) fp32.  This is the (m, l, O) a rank of the
 * page's kernel sends toward the root; gqa_merge folds several of them. */
gqa_status gqa_decode_partial(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                              float* m, float* l, float* o_part,
                              int batch, int T_q, int64_t S_kv, int64_t s_begin, int64_t s_len,
                              int h_q, int h_kv, int d_head, float scale,
                              void* workspace, size_t ws_bytes, void* stream);

gqa_status gqa_decode_partial_ex(const uint16_t* q, const uint16_t* k, const uint16_t* v,
                                 float* m, float* l, float* o_part,
                                 int batch, int T_q, int64_t S_kv, int64_t s_begin, int64_t s_len,
                                 int h_q, int h_kv, int d_head, float scale,
                                 void* workspace, size_t ws_bytes, void* stream,
                                 const gqa_options* opt);

/* Merge n_parts >= 1 partials laid out m, l: [n_parts][rows], o_part: [n_parts][rows][d_head]
 * (page: _merge_running folded over the parts, then O / l), writing
 * o (rows, d_head) f16.  Rows whose partials are all empty (m = -inf) give 0. */
gqa_status gqa_merge(const float* m, const float* l, const float* o_part, int n_parts,
                     int64_t rows, int d_head, uint16_t* o, void* stream);

/* gqa_merge with options: gqa_options.bf16 writes o as bfloat16 instead of IEEE binary16 (the
 * other fields are not used).  opt NULL = gqa_merge. */
gqa_status gqa_merge_ex(const float* m, const float* l, const float* o_part, int n_parts,
                        int64_t rows, int d_head, uint16_t* o, void* stream, const gqa_options* opt);

/* As gqa_merge but keeps the merged partial (one hop of the page's chain reduce):
 * m_out, l_out (rows) and o_out (rows, d_head), fp32. */
gqa_status gqa_merge_partial(const float* m, const float* l, const float* o_part, int n_parts,
                             int64_t rows, int d_head, float* m_out, float* l_out, float* o_out,
                             void* stream);

/* Paged decode (page "muh_kernel_map.py", paged_attention_v2 shape; T_q = 1).
 *   q             (num_seqs, h_q*d_head) f16
 *   k_pool/v_pool (num_blocks, block_size, h_kv*d_head) f16: token j of sequence b is row
 *                 j % block_size of block block_tables[b, j / block_size]
 *   block_tables  (num_seqs, max_blocks_per_seq) int32; entries past a sequence's last block
 *                 are never read
 *   seq_lens      (num_seqs) int32 in [0, min(max_seq_len, max_blocks_per_seq*block_size)];
 *                 a length-0 sequence gets O = 0
 *   o             (num_seqs, h_q*d_head) f16, written
 * block_size in {8, 16, 32, 64}; partition_size a multiple of 64 with
 * partition_size / min(block_size, 16) <= 1024, or 0 = automatic (the page's v2: 512-token
 * partitions, a partition pass and a merge pass).  A partition_size of at least max_seq_len is
 * the page's single-pass v1 (page "muh_kernel_map.py", paged_attention_v1, for seq_len <= 8192):
 * one pass over each whole sequence and no merge launch; on GB300 it measured no faster than v2
 * on any batch tried, so the automatic choice does not take it.  max_seq_len (host-known bound
 * on seq_lens) sizes the grid.  Block ids outside [0, num_blocks) are not loaded and are
 * reported by gqa_workspace_check. */
gqa_status gqa_decode_paged(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                            const int32_t* block_tables, const int32_t* seq_lens, uint16_t* o,
                            int num_seqs, int max_blocks_per_seq, int num_blocks, int block_size,
                            int partition_size, int h_q, int h_kv, int d_head, float scale,
                            int max_seq_len, void* workspace, size_t ws_bytes, void* stream);

gqa_status gqa_decode_paged_ex(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                               const int32_t* block_tables, const int32_t* seq_lens, uint16_t* o,
                               int num_seqs, int max_blocks_per_seq, int num_blocks, int block_size,
                               int partition_size, int h_q, int h_kv, int d_head, float scale,
                               int max_seq_len, void* workspace, size_t ws_bytes, void* stream,
                               const gqa_options* opt);

/* Paged decode over vLLM's cache layout (page "muh_kernel_map.py", VLLM_KERNEL_MAP
 * 'paged_attention_v1': key_cache [num_blocks, num_kv_heads, head_dim/x, block_size, x]), read in
 * place.  x = 8 (16-byte vectors of 16-bit elements).  The page gives no value-cache layout; the
 * same serving stack's [num_blocks, num_kv_heads, head_dim, block_size] is taken:
 *   k_cache  (num_blocks, h_kv, d_head/8, block_size, 8) f16 / bf16
 *   v_cache  (num_blocks, h_kv, d_head, block_size)      f16 / bf16
 * Everything else -- q, block_tables, seq_lens, o, partition_size (0 = automatic, 512),
 * workspace (gqa_paged_workspace_size), options, errors -- as gqa_decode_paged, except that a
 * work item's KV heads (gqa_options.paged_head_group) are at most 64 / block_size (a TMA box
 * holds whole blocks; the automatic choice respects it).  Additionally
 * num_blocks * h_kv * d_head / 8 must be < 2^31. */
gqa_status gqa_decode_paged_vllm(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                 const int32_t* block_tables, const int32_t* seq_lens, uint16_t* o,
                                 int num_seqs, int max_blocks_per_seq, int num_blocks, int block_size,
                                 int partition_size, int h_q, int h_kv, int d_head, float scale,
                                 int max_seq_len, void* workspace, size_t ws_bytes, void* stream);

gqa_status gqa_decode_paged_vllm_ex(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                                    const int32_t* block_tables, const int32_t* seq_lens, uint16_t* o,
                                    int num_seqs, int max_blocks_per_seq, int num_blocks, int block_size,
                                    int partition_size, int h_q, int h_kv, int d_head, float scale,
                                    int max_seq_len, void* workspace, size_t ws_bytes, void* stream,
                                    const gqa_options* opt);

/* Size of the per-GPU device array used by gqa_decode_noalloc: 8 MiB. */
#define GQA_NOALLOC_SCRATCH_BYTES (8u * 1024u * 1024u)

/* gqa_decode for callers that cannot allocate device memory -- e.g. a plugin whose device
 * memory is budgeted by its host framework, a latency-critical loop that cannot afford
 * cudaMalloc's implicit synchronisation, or a C / FFI caller with no device allocator.
 * No counterpart on the pages: it is the same decode step with the workspace replaced by a
 * library-owned device array of GQA_NOALLOC_SCRATCH_BYTES on every GPU that loads the
 * library (held until the process exits).  The caller still passes q, k, v and o as for
 * gqa_decode.  The call allocates nothing.
 *  - Shapes whose workspace (gqa_decode_workspace_size with n_splits = 0) exceeds
 *    GQA_NOALLOC_SCRATCH_BYTES are rejected with GQA_ERR_WORKSPACE; use gqa_decode then.
 *  - The first call on each device looks up the array's device address
 *    (cudaGetSymbolAddress) with that device current; make that first call before any
 *    stream capture.
 *  - Every call on a device shares the one array: calls that overlap on the GPU (other
 *    streams, other host threads) race and corrupt each other's results.  Each call
 *    clears the array's arrival counters on `stream` before its kernel.
 *  - Faults seen on the device (a bounded wait that gave up) set bits in the array's status
 *    word, which calls do not clear: they accumulate until gqa_decode_noalloc_check reads
 *    them.  Outputs of calls made since the last clean check are then invalid. */
gqa_status gqa_decode_noalloc(const uint16_t* q, const uint16_t* k, const uint16_t* v, uint16_t* o,
                              int batch, int T_q, int64_t S_kv, int h_q, int h_kv, int d_head, float scale,
                              void* stream);

/* The status word of the current device's gqa_decode_noalloc array: synchronise `stream`, read
 * and clear it.  GQA_OK, or GQA_ERR_TIMEOUT (a bounded device wait gave up in some call since the
 * last check; those outputs are invalid).  Allocates nothing.  Like gqa_decode_noalloc, it must
 * not overlap other calls on the same device. */
gqa_status gqa_decode_noalloc_check(void* stream);

#ifdef __cplusplus
}
#endif

#endif /* GQA_DECODE_H_ */
