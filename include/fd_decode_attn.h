/*
 * fd_decode_attn.h - C ABI of libfd.so: single-token split-KV decode attention
 * (Flash-Decoding) over a position-addressed bf16 KV cache, for NVIDIA GB300
 * (sm_103a).
 *
 * What the library computes is defined in "Hand-Writing Gemma 4
 * Flash-Decoding + an FP4 Matvec Bonus (Part 2)", section "One KV head breaks
 * the textbook": one query token per sequence attends over its KV cache with
 * GQA/MQA grouping; the kernel walks absolute positions, reading position pos
 * from slot pos % capacity, and reads only the live band
 * [max(0, len - window), len); the key sequence is split across thread blocks
 * whose unnormalised (O, m, l) partials are combined by an online-softmax
 * merge ("fixup") kernel. For every sequence b and query head h:
 *
 *     kvh   = h / (NH / NKV)
 *     band  = [max(0, len_b - min(W, capacity)), len_b),  W = window or infinity
 *     s_p   = scale * dot(q[b][h], K[b][kvh][p % capacity])   for p in band
 *     out[b][h] = sum_p softmax(s)_p * V[b][kvh][p % capacity]
 *
 * len_b == 0 gives an all-zero output row.
 *
 * Conventions shared by every entry point:
 *   - Return value: FD_OK (0) or one of the FD_ERR_* codes below. No C++
 *     exception crosses this boundary. On any error nothing is launched.
 *   - All tensors are caller-owned DEVICE memory of the current CUDA device,
 *     row-major, densely packed:
 *       q        bf16  [B][NH][HS]          (= [B, 1, NH*HS]; Q head h of
 *                                            group kvh is row kvh*G + h%G)
 *       k_cache  bf16  [B][NKV][capacity][HS]   position p of sequence b lives
 *       v_cache  bf16  [B][NKV][capacity][HS]   in row (b, kvh, p % capacity)
 *       out      bf16  [B][NH][HS]          rounded to nearest even
 *       out_f32  fp32  [B][NH][HS]          optional copy before rounding
 *       lens     int32 [B]                  len_b, counting the current token
 *     q, k_cache, v_cache, out, out_f32 and the workspace must be 16-byte
 *     aligned, lens 4-byte aligned (else FD_ERR_ALIGNMENT).
 *   - Supported shapes: HS in {64, 128, 256, 512}; NH % NKV == 0 and
 *     G = NH / NKV <= 16; capacity >= 1; window <= 0 means no window, and
 *     window > capacity is rejected (FD_ERR_INVALID_ARG). B == 0 is a no-op.
 *   - scale <= 0 selects 1/sqrt(HS) (the attnScale convention of
 *     SharpInference issue #156, "Background").
 *   - Launches are asynchronous on `stream`; no entry point that launches
 *     work synchronises the host, so a call can be captured in a CUDA graph
 *     once its workspace exists. `lens` is read on the device, so replays of
 *     a captured call see the current lengths.
 *   - Lengths that break the cache's precondition are repaired on the device
 *     and reported through the device error word (fd_get_device_error):
 *     len_b < 0 is treated as 0; with no window, len_b > capacity keeps the
 *     last `capacity` positions.
 */
#ifndef FD_DECODE_ATTN_H_
#define FD_DECODE_ATTN_H_

#include <stddef.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Same type as cudaStream_t; NULL is the legacy default stream. */
typedef struct CUstream_st* fd_stream_t;

enum {
  FD_OK = 0,
  FD_ERR_INVALID_ARG = 1,   /* null pointer, bad size, window > capacity, bad plan */
  FD_ERR_UNSUPPORTED = 2,   /* HS not in {64,128,256,512}, NH % NKV != 0, G > 16 */
  FD_ERR_ALIGNMENT = 3,     /* a pointer is not aligned as required */
  FD_ERR_CUDA = 4,          /* a CUDA runtime call or a launch failed */
  FD_ERR_WORKSPACE = 5,     /* workspace too small, or would need allocating during capture */
  FD_ERR_SCRATCH_LIMIT = 6  /* fd_decode_attn_noalloc: the shape needs more than its fixed scratch */
};

/* Size of the fixed device scratch array behind fd_decode_attn_noalloc. */
#define FD_NOALLOC_SCRATCH_BYTES (32u << 20)

/* Bits of the device error word (fd_get_device_error). */
enum {
  FD_DEVERR_LEN_NEGATIVE = 1u << 0,  /* some len_b < 0; treated as 0 */
  FD_DEVERR_LEN_CLAMPED = 1u << 1,   /* no window and len_b > capacity; band clamped */
  FD_DEVERR_WAIT_TIMEOUT = 1u << 2,  /* a pipeline wait gave up; the output is invalid */
  FD_DEVERR_MIN_LEN = 1u << 3        /* some len_b < the plan's min_len: slots outside the live band
                                        may have been read early (the output is still exact) */
};

/* KV cache element types (fd_plan_t.kv_dtype). */
enum {
  FD_KV_BF16 = 0,  /* bf16 K and V: fd_decode_attn, fd_decode_attn_ex, fd_decode_attn_noalloc */
  FD_KV_E4M3 = 1   /* FP8 E4M3 codes with fp32 scales: fd_decode_attn_fp8, fd_decode_attn_fp8_ex */
};

/* Kernel families. */
enum {
  FD_PATH_AUTO = 0,   /* let the plan choose */
  FD_PATH_SIMT = 1,   /* plain per-position fp32 kernel; reference GPU path */
  FD_PATH_TC = 2,     /* bulk-copy pipelined, tensor-core (mma) tile kernel */
  FD_PATH_UMMA = 3    /* TMA + tcgen05 kernel, accumulators in tensor memory: bf16,
                         HS 512, 8 < G <= 16, window <= 0 */
};

/*
 * Launch plan: how many key-sequence splits each (sequence, KV head) gets,
 * how the split blocks are grouped into thread-block clusters, and how much
 * workspace the partials need. Built by fd_plan / fd_plan_sms; the caller may
 * change num_splits, path and cluster through fd_plan_override only.
 *
 * Split rule (the page gives none; "One KV head breaks the textbook" only says
 * to split the key sequence across blocks so one KV head still fills the GPU):
 * units U = B * NKV; enough splits that U * num_splits covers every CTA slot of
 * the GPU once; a split then never exceeds `max_chunk` positions (a bound that
 * keeps ragged batches balanced), rounding num_splits up to a whole number of
 * waves when that bound applies. Where filling the GPU would cut the band
 * into pieces under two tiles of the tensor-core kernel, chunks are whole
 * tiles (`granule` = the tile's positions: a split shorter than a tile costs
 * a full tile's latency and adds a partial), so a short band gets fewer
 * splits; otherwise the granule is 1. An E4M3 cache with head dim 64 or 128
 * then uses a half-length tile (1 KB copy groups: 128 or 64 positions). With
 * no window, or a window as long as the cache, a band occupies slots
 * [0, band) and the tensor-core kernel deals its tiles to the splits in turn
 * (split s: tiles s, s + S, ...) instead of cutting chunks. On
 * the device each sequence cuts its own band into chunks of
 * ceil(band_b / num_splits) positions rounded up to the granule, so a short
 * sequence uses fewer, not emptier, splits.
 *
 * With G >= 8 query rows per KV head a partial (G x HS floats) is costly
 * next to a split's K/V bytes, and the plan fills each SM once instead of
 * with every resident block, unless that would put more than ~2 MiB of K+V
 * in a split: then it fills every resident block slot once, with up to
 * ~4 MiB per split, before adding waves.
 *
 * Fused merge (opt-in through fd_plan_override; plans use fused = 0), two
 * forms, neither launching the merge kernel:
 *   fused = 1, the last block: when a group's partials are small
 *   (G * S * HS * 4 bytes <= 256 KB), the last split block of each (sequence,
 *   KV head) to finish merges them itself, found with a per-group counter
 *   (one acquire-release atomic per block) that wraps back to zero.
 *   fused = 2, the group step: when the whole grid is resident at once
 *   (B * NKV * S <= num_sms * ctas_per_sm), the grid is launched
 *   cooperatively; every active split block of a group counts in on the same
 *   counter, waits (bounded) until the whole group has, then merges its
 *   share of the group's G x HS outputs, and counts out on a second word
 *   (B * NKV more workspace words after the counters); the last block out
 *   sets both back to zero.
 *
 * Copy groups: a tile's K and V rows arrive in groups of about 2 KB, one
 * bulk copy per group. Head dim 256 with at most 8 query rows per KV head
 * (the sliding ring) uses 4 KB groups (64-position tiles; one pipeline stage
 * when every split of the plan is at most one tile, else two). For head dim
 * 512 with more than 8 query rows per KV head, when the whole grid fits one
 * wave at one block per SM, the plan uses 4 KB groups too: fewer copies per
 * block, and a block's copy rate is set by its copy count.
 *
 * Tensor-memory kernel (opt-in through fd_plan_override(..., FD_PATH_UMMA, ...);
 * plans never choose it): for the MQA geometry of "One KV head breaks the
 * textbook" (bf16, HS 512, 8 < G <= 16, window <= 0) each split block takes a
 * consecutive slice of the band's slots [0, min(len, capacity)) in chunks of
 * 16 positions (granule 16), streams K and V through one shared-memory ring
 * of 32 KB slots as TMA boxes of 128/64/32/16/8 rows in the order K(0), then
 * V(i) and K(i + 1) alternately (the last rows of the band that do not fill 8
 * are loaded by the copy warp, so exactly the band is read), and one thread
 * issues S^T = K Q^T and O^T += V^T P^T as tcgen05 MMAs with the accumulators
 * in tensor memory, the next tile's scores while the current tile's softmax
 * runs. Such a plan has group_bytes = 16384 (one TMA box), consumer_warps = 4,
 * cluster = 1 and no fused merge; the merge kernel is the same. Measured on
 * GB300: level with FD_PATH_TC on long MQA bands, slower on short ones.
 *
 * Clusters (opt-in through fd_plan_override; plans use cluster = 1): the
 * blocks of `cluster` consecutive splits form a thread-block cluster and
 * combine their partials through distributed shared memory, so only
 * num_splits / cluster partials per row reach the workspace; when
 * cluster == num_splits one cluster covers the whole band and writes the
 * output itself (no merge kernel, no workspace).
 */
typedef struct {
  int num_splits;          /* S: grid splits per (sequence, KV head) */
  int path;                /* FD_PATH_SIMT, FD_PATH_TC or FD_PATH_UMMA */
  int cluster;             /* blocks per cluster along the splits; divides S; 1 = none */
  int granule;             /* chunk rounding on the device, positions: 1, or the tile for short bands; 16 for FD_PATH_UMMA */
  int max_band;            /* band bound the plan was sized for */
  int ctas_per_sm;         /* resident CTAs per SM the plan assumed */
  int num_sms;             /* SM count the plan assumed */
  int max_cluster;         /* largest cluster the device schedules for this kernel */
  int fused;               /* 1: each group's last split block merges; 2: the group step (no merge kernel) */
  int group_bytes;         /* bytes per bulk-copy group of a tile: 2048 or 4096 (bf16); 2048 or 1024 (E4M3) */
  int kv_dtype;            /* FD_KV_BF16 or FD_KV_E4M3: the cache type the plan was made for */
  int consumer_warps;      /* MMA warps per split block (2, 4 or 8; 0 on the SIMT path) */
  int persistent;          /* blocks of a persistent split grid (fd_plan_persistent); 0: one block per split */
  int min_len;             /* caller's lower bound on every len_b (fd_plan_min_len); 0: none */
  size_t workspace_bytes;  /* bytes of workspace fd_decode_attn_ex needs */
  size_t workspace_zero_bytes; /* leading workspace bytes that must be zero before first use */
  /* the shape the plan was made for; fd_decode_attn_ex checks it */
  int B, NH, NKV, HS, capacity, window;
} fd_plan_t;

/*
 * fd_plan: build a plan for the given shape on CUDA device `device` (its SM
 * count and the kernel's occupancy are queried). max_len > 0 bounds len_b
 * (tighter plans for short contexts); max_len <= 0 uses the largest band the
 * cache can hold, min(window, capacity). Pure host computation plus device
 * attribute queries; launches nothing and allocates nothing.
 * Errors: FD_ERR_INVALID_ARG, FD_ERR_UNSUPPORTED, FD_ERR_CUDA (query failed).
 */
int fd_plan(int B, int NH, int NKV, int HS, int capacity, int window, int max_len,
            int device, fd_plan_t* plan);

/*
 * fd_plan_sms: the same plan for a GPU with `num_sms` SMs, `ctas_per_sm`
 * resident CTAs per SM and clusters of at most `max_cluster` blocks, without
 * touching any device (for tools and tests).
 */
int fd_plan_sms(int B, int NH, int NKV, int HS, int capacity, int window, int max_len,
                int num_sms, int ctas_per_sm, int max_cluster, fd_plan_t* plan);

/*
 * fd_plan_kv / fd_plan_sms_kv: fd_plan / fd_plan_sms for a cache of element
 * type kv_dtype (FD_KV_BF16 gives the same plan as fd_plan / fd_plan_sms).
 * An E4M3 plan runs on FD_PATH_TC only and bounds a split by the same ~2 MiB
 * of K+V bytes, so its splits may hold twice the positions. Its copy groups
 * are 2 KB (1 KB for head dim 256 with more than 8 query rows, and for the
 * half-length tiles above) and its head-dim-512, 16-row tile uses
 * eight consumer warps when the grid is one block per SM, four otherwise
 * (measured on GB300: copy count per block and issue slots per SM).
 * Errors: FD_ERR_INVALID_ARG (unknown kv_dtype), those of fd_plan / fd_plan_sms.
 */
int fd_plan_kv(int B, int NH, int NKV, int HS, int capacity, int window, int max_len,
               int device, int kv_dtype, fd_plan_t* plan);
int fd_plan_sms_kv(int B, int NH, int NKV, int HS, int capacity, int window, int max_len,
                   int num_sms, int ctas_per_sm, int max_cluster, int kv_dtype, fd_plan_t* plan);

/*
 * fd_plan_override: force the split count (num_splits >= 1; 0 keeps the
 * plan's), the kernel family (path != FD_PATH_AUTO; FD_PATH_UMMA only for the
 * shapes above), the cluster size
 * (cluster >= 1, a power of two <= 16 that divides num_splits and HS / 4;
 * 0 keeps the plan's; the SIMT path takes cluster 1 only) and/or the fused
 * merge (fused = 0 off, 1 the last block, 2 the group step, each where
 * allowed; -1 the plan's rule), then
 * recompute the dependent fields (fused, group_bytes, workspace sizes). Used
 * to test that the result does not depend on these choices, and to bisect.
 * Errors: FD_ERR_INVALID_ARG.
 */
int fd_plan_override(fd_plan_t* plan, int num_splits, int path, int cluster, int fused);

/*
 * fd_plan_persistent: run the split kernel as a persistent grid (persistent =
 * 1), as one block per split (0), or as the plan's rule decides (-1).
 * "Hand-Writing Gemma 4 Flash-Decoding + an FP4 Matvec Bonus (Part 2)",
 * section "One KV head breaks the textbook", gives each (KV head, split) its
 * own block; a persistent grid keeps one block per resident block slot
 * (plan->persistent = min(work items, num_sms * ctas_per_sm)) and hands out the
 * work items (split, KV head, sequence), longest bands first as in the
 * one-block-per-split order, from a 32-bit counter in the workspace. A block's
 * copy warps stream the next item's first tiles while its MMA warps finish the
 * current one, so the pipeline does not drain and refill between items. The
 * counter wraps back to zero when the last block takes its final index, so the
 * workspace stays reusable. Tensor-core path only, without clusters or the
 * fused merge; fd_plan_override resets the choice to the plan's rule, and
 * plans use persistent = 0 (on GB300 it gained at most ~1% on multi-wave
 * grids and lost on one-wave grids). The result is bit-identical to one
 * block per split (the same partials, merged in the same order).
 * Errors: FD_ERR_INVALID_ARG (bad plan or mode, or persistent = 1 where it is
 * not available).
 */
int fd_plan_persistent(fd_plan_t* plan, int persistent);

/*
 * fd_plan_min_len: record that every len_b the plan will be used with is at
 * least min_len (>= 0; 0, the plans' default, promises nothing). The live band
 * is read only: a split block reads nothing before it has read its sequence's
 * length, except the tiles of slots that every length >= min_len makes live.
 * With no window, or a window as long as the cache, the band's slots are
 * [0, min(len_b, capacity)), so the slots [0, min(min_len, capacity)) are live
 * for any such length; the tensor-core kernel asks L2 for this split's such
 * tiles while the previous kernel on the stream still runs, and copies its
 * first ones as soon as that kernel is done, before its length arrives
 * ("Hand-Writing Gemma 4 Flash-Decoding + an FP4 Matvec Bonus (Part 2)",
 * section "One KV head breaks the textbook": reads only the live band, never
 * the allocation). A decode loop's host knows its lengths, so it can pass the
 * smallest; a full sliding ring (len_b >= capacity) passes capacity. A length
 * below the bound still gives the exact result (tiles read early and not in
 * the band are never used) and raises FD_DEVERR_MIN_LEN.
 * Errors: FD_ERR_INVALID_ARG (null plan, min_len < 0).
 */
int fd_plan_min_len(fd_plan_t* plan, int min_len);

/*
 * fd_workspace_bytes: workspace a plan needs. With P = num_splits / cluster
 * partial slots per row: when P > 1, B * NKV 32-bit split counters (twice
 * that with the group step, fused = 2); with a
 * persistent grid, one more 32-bit work-item counter; when P > 1, then
 * B * NH * P * HS fp32 partial outputs and B * NH * P * 2 fp32 (m, l). Each
 * part is rounded up to 256 bytes. 0 when P == 1 without a persistent grid
 * (the split kernel then writes the output itself). The counters (the first
 * workspace_zero_bytes bytes) must be zero before a workspace's first use;
 * every completed call leaves them zero (after a call that reported
 * FD_DEVERR_WAIT_TIMEOUT, clear them again).
 */
size_t fd_workspace_bytes(const fd_plan_t* plan);

/*
 * fd_decode_attn: the whole hot path in one call - split kernel, then merge
 * kernel - with a plan made for the current device (max_len <= 0) and a
 * workspace the library owns, one per (device, stream), grown on demand and
 * kept until fd_release. The first call for a (device, stream) and shape
 * allocates with cudaMalloc (which synchronises the device) and must not be
 * made while the stream is being captured; later calls with shapes needing no
 * more workspace allocate nothing and may be captured. Capture with a
 * too-small workspace returns FD_ERR_WORKSPACE.
 * Errors: every FD_ERR_* code.
 */
int fd_decode_attn(const void* q, const void* k_cache, const void* v_cache, void* out,
                   const int* lens, int B, int NH, int NKV, int HS, int capacity,
                   int window, float scale, fd_stream_t stream);

/*
 * fd_decode_attn_ex: the same with an explicit plan, a caller-owned device
 * workspace of workspace_bytes >= fd_workspace_bytes(plan) whose first
 * plan->workspace_zero_bytes bytes were zero before its first use (every
 * completed call leaves them zero; the rest is scratch between calls; calls
 * that overlap on the GPU must not share one), and an optional fp32 copy of
 * the output (out_f32 may be NULL). The shape arguments must equal the plan's.
 * Allocates nothing.
 * Errors: every FD_ERR_* code.
 */
int fd_decode_attn_ex(const fd_plan_t* plan, void* workspace, size_t workspace_bytes,
                      float* out_f32, const void* q, const void* k_cache,
                      const void* v_cache, void* out, const int* lens, int B, int NH,
                      int NKV, int HS, int capacity, int window, float scale,
                      fd_stream_t stream);

/*
 * fd_decode_attn_fp8 / fd_decode_attn_fp8_ex: the same attention over an FP8
 * cache. "Hand-Writing Gemma 4 Flash-Decoding + an FP4 Matvec Bonus
 * (Part 2)": the paragraph on the open problem just before section "What we'd
 * tell the next person" leaves the long-band MQA latency residual to FP8 KV
 * storage, which halves the bytes per position; that section adds that FP8
 * KV needs no special hardware, the values being widened inline where they
 * are used. Reading taken (the page fixes no scale granularity): one fp32
 * scale per (sequence, KV head) for K and one for V.
 *     k8, v8    uint8 [B][NKV][capacity][HS]  E4M3 codes (1 sign, 4 exponent
 *                                             bits with bias 7, 3 mantissa
 *                                             bits; no infinity; x111_1111 NaN)
 *     k_scale   fp32  [B][NKV]   K[b][kvh][slot][d] = E4M3(k8[...]) * k_scale[b][kvh]
 *     v_scale   fp32  [B][NKV]   the same for V
 * q, out, out_f32, lens and every other convention are those of
 * fd_decode_attn / fd_decode_attn_ex; k8 and v8 must be 16-byte aligned and
 * the scales 4-byte aligned. Arithmetic: every E4M3 value is an fp16 value,
 * so codes widen to fp16 exactly; q is scaled by a power of two per block
 * (exact) and rounded to fp16 (exact for bf16 inputs within a factor 2^30
 * of the block's largest |q|); products accumulate in fp32; the softmax weights
 * enter the P.V product as fp16 (relative error at most 2^-11 per weight);
 * O is multiplied by the V scale once at the end. fd_decode_attn_fp8_ex needs
 * an FD_KV_E4M3 plan (fd_plan_kv) and the bf16 entry points an FD_KV_BF16
 * plan; a plan of the other type is FD_ERR_INVALID_ARG. Workspace: as for
 * fd_decode_attn / fd_decode_attn_ex (fd_decode_attn_fp8 shares the
 * library-owned workspaces).
 * Errors: every FD_ERR_* code.
 */
int fd_decode_attn_fp8(const void* q, const void* k8, const void* v8, const float* k_scale,
                       const float* v_scale, void* out, const int* lens, int B, int NH,
                       int NKV, int HS, int capacity, int window, float scale,
                       fd_stream_t stream);
int fd_decode_attn_fp8_ex(const fd_plan_t* plan, void* workspace, size_t workspace_bytes,
                          float* out_f32, const void* q, const void* k8, const void* v8,
                          const float* k_scale, const float* v_scale, void* out,
                          const int* lens, int B, int NH, int NKV, int HS, int capacity,
                          int window, float scale, fd_stream_t stream);

/*
 * fd_decode_attn_noalloc: the same computation as fd_decode_attn, for callers
 * that must not allocate device memory while they run (for example an op
 * inside a serving framework whose memory pool owns the device, or a
 * latency-critical decode loop in which cudaMalloc could synchronise the
 * device or fail mid-step). It allocates nothing: the split partials live in
 * a fixed file-scope device array of FD_NOALLOC_SCRATCH_BYTES (32 MiB) that
 * every device using the library holds until the process exits. There is no
 * counterpart on the pages; it is an addition of this library.
 *   - Same arguments, layouts and conventions as fd_decode_attn; the plan is
 *     made for the current device with max_len <= 0.
 *   - The array holds, in its first 64 KB, the counters a plan keeps at the
 *     head of its workspace (plan->workspace_zero_bytes: one 32-bit split
 *     counter per (sequence, KV head), rounded up to 256 bytes), and the
 *     partials in the rest. A shape whose plan needs more
 *     (workspace_zero_bytes > 64 KB, i.e. B * NKV > 16384, or more than
 *     32 MiB - 64 KB of partials) is rejected with FD_ERR_SCRATCH_LIMIT
 *     before anything is launched (fd_plan + fd_workspace_bytes tell in
 *     advance).
 *   - The first call on a device looks up the array's device address on that
 *     device (cudaGetSymbolAddress), clears the array with cudaMemsetAsync on
 *     `stream`, waits for `stream` (once, so the clear has finished before any
 *     call on any stream runs), and caches the address.
 *   - All calls on a device share the one array and each finds the previous
 *     call's contents in it. The counters must start at zero: the device's
 *     set-up clears the array once and every completed call leaves them zero.
 *     A call that returned FD_ERR_CUDA, or after which fd_get_device_error
 *     reported FD_DEVERR_WAIT_TIMEOUT, may leave a counter non-zero: call
 *     fd_release, and the next call on each device clears the array again.
 *     Calls that overlap on the GPU - other streams, other threads - race on
 *     it: the caller must serialise them.
 * Errors: every FD_ERR_* code.
 */
int fd_decode_attn_noalloc(const void* q, const void* k_cache, const void* v_cache, void* out,
                           const int* lens, int B, int NH, int NKV, int HS, int capacity,
                           int window, float scale, fd_stream_t stream);

/*
 * fd_debug_withhold_copies: a test hook for the bounded waits (no counterpart
 * on the pages). With withhold_tile >= 0, the tensor-core split blocks of
 * every later call on any device issue no K/V copies for their tiles from
 * index withhold_tile on (they never issue those copies, so nothing is left
 * in flight), the consumer warps' wait for that tile gives up after
 * wait_limit_ns nanoseconds (0: the default, about one second), the call
 * completes with an invalid output, and fd_get_device_error reports
 * FD_DEVERR_WAIT_TIMEOUT; the workspace counters may then be non-zero.
 * withhold_tile < 0 restores normal operation and the default limit. Sets the
 * limit on the current device (a synchronous copy); not for use while other
 * threads call the library.
 * Errors: FD_ERR_CUDA.
 */
int fd_debug_withhold_copies(int withhold_tile, unsigned long long wait_limit_ns);

/*
 * fd_get_device_error: wait for `stream`, then return in *err the OR of the
 * FD_DEVERR_* bits raised on the current device since the last read, and
 * clear them. Synchronises the host: for tests and diagnostics only.
 * Errors: FD_ERR_INVALID_ARG (err NULL), FD_ERR_CUDA.
 */
int fd_get_device_error(fd_stream_t stream, unsigned int* err);

/* fd_release: free the library-owned workspaces of every device, and make
 * the next fd_decode_attn_noalloc call on each device clear its scratch array
 * again (the recovery step after a failed call). Not thread-safe against
 * concurrent calls of the library. */
void fd_release(void);

/* fd_strerror: static, human-readable text for an FD_* status code. */
const char* fd_strerror(int status);

/* fd_version: (major << 16) | (minor << 8) | patch. */
int fd_version(void);

#ifdef __cplusplus
}
#endif

#endif /* FD_DECODE_ATTN_H_ */
