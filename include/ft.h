/*
 * ft.h -- C ABI of a GB300-native routed-expert cache for MoE layers.
 *
 * The full routed-expert pool lives in pinned host memory (the source of truth);
 * HBM holds a global, cross-layer cache of whole (layer, expert) slots.
 *
 * Pages cited (by title; sections as printed on each page):
 *   [EXPLAINER] "FreeToken: Efficient Edge-Native MoE Serving with Bandwidth-Adaptive
 *               Execution" (blog explainer of the arXiv v1 paper)
 *   [QIITA]     "FreeTokenってなんだ？ ─ 8GBノートPCで35Bを動かす判断基準"
 *   [BWRATIO]   "FreeToken hybrid MoE 后端：带宽比如何决定专家「搬」还是「算」"
 *   [JUHE]      the juhe.plus article on FreeToken's 8 GB RTX 4060 Laptop result
 *               (cited by its section headings)
 *
 * Conventions
 *   - Every call returns ft_status; FT_OK is 0.  No C++ exception crosses the ABI.
 *   - The caller owns all memory: the host pool, the slot buffer, the workspace,
 *     inputs and outputs.  The library owns only the opaque ft_cache handle, one
 *     internal copy stream and CUDA events.
 *   - `stream` arguments are cudaStream_t values passed as void* (NULL = legacy
 *     default stream).  Per-token calls (ft_moe_decode) are asynchronous on it,
 *     perform no host synchronisation and no allocation.
 *   - Pointers marked "device" must be device (or managed) memory of the current
 *     device; "host" pointers are ordinary host memory; "pinned" means allocated
 *     with ft_pinned_alloc or otherwise page-locked and mapped.
 *   - Sizes are element counts unless they end in _bytes.
 *
 * Record layout (one per flat id l*E + e; see ft_record_bytes):
 *   [W_gu codes 2I*H/2][W_gu scales 2I*H/16][W_d codes H*I/2][W_d scales H*I/16]
 *   [s_gu fp32][s_d fp32], padded to a multiple of 256 bytes.
 *   W_gu is [2I, H] row-major (gate rows 0..I-1, up rows I..2I-1); W_d is [H, I].
 *   NVFP4: E2M1 codes, two per byte with element 2j in the low nibble; one unsigned
 *   E4M3 scale per 16 consecutive elements of a row; one fp32 tensor scale per
 *   matrix.  value = e2m1(code) * e4m3(scale) * s_t.
 */
#ifndef FT_H
#define FT_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef int32_t ft_status;
#define FT_OK            0
#define FT_ERR_ARG       1   /* bad argument (size, layer, pointer, id range) */
#define FT_ERR_CUDA      2   /* a CUDA runtime call failed */
#define FT_ERR_CAPACITY  3   /* not enough slots for the requested operation */
#define FT_ERR_STATE     4   /* call not allowed in the current state (e.g. capturing) */
#define FT_ERR_TIMEOUT   5   /* a bounded device wait ran out */
#define FT_ERR_UNPINNED  6   /* host pool is not page-locked / mapped */

/* Bits of the device status word (ft_cache_status). */
#define FT_DEV_BAD_ID    0x1 /* a route id outside [0, E) was masked */
#define FT_DEV_TIMEOUT   0x2 /* a bounded device wait ran out */
#define FT_DEV_SCALE_RANGE 0x4 /* prefill of MXFP4 experts: a block scale outside
                                  2^-9..2^8 has no exact UE4M3 twin (clamped) */

/* Expert record formats ([EXPLAINER §9.2]: NVFP4 on the NVFP4 machines; DeepSeek-V4-
 * Flash's routed experts are natively MXFP4 and are consumed bit-exactly).
 * FT_FORMAT_NVFP4: E2M1 codes, unsigned E4M3 scale per 16 elements, fp32 tensor scale
 *   per matrix (the record layout above).
 * FT_FORMAT_MXFP4: E2M1 codes, E8M0 scale per 32 elements (value 2^(c-127)); same
 *   layout with the scale arrays [rows, K/32]; the two tensor-scale words are 1.0. */
#define FT_FORMAT_NVFP4 0
#define FT_FORMAT_MXFP4 1

typedef struct ft_cache ft_cache;

/* Miss split ([EXPLAINER §6.2-6.5]; [BWRATIO "第二层带宽比"]).
 * FT_SPLIT_FULL_OFFLOAD: every unique miss is filled (q = m).
 * FT_SPLIT_QSTAR: q follows the Q16 integer rule of [BWRATIO "代码全链路" §3] with
 *   f_q16 in [1, 65536], then q >= 1 ([EXPLAINER §6.5]), then q <= C - |H|. */
#define FT_SPLIT_FULL_OFFLOAD 0
#define FT_SPLIT_QSTAR        1
typedef struct {
    int32_t  mode;
    uint32_t f_q16;
} ft_split;

typedef struct {
    int32_t L;              /* MoE layers */
    int32_t E;              /* routed experts per layer (1..4096) */
    int32_t H;              /* hidden size, multiple of 64, at most 8192 */
    int32_t I;              /* expert intermediate size, multiple of 32, at most 4096 */
    int32_t k_max;          /* largest top-k passed to ft_moe_decode (1..32) */
    int32_t B_max;          /* largest decode batch (1..32) */
    int32_t capacity;       /* slots C at creation (1..16384) */
    int32_t capacity_max;   /* largest C ever used by ft_cache_resize (0 = capacity) */
    int32_t T_max;          /* largest prefill chunk in tokens (0 = no prefill) */
    const void* host_pool;  /* pinned, L*E records of ft_record_bytes(H, I) bytes */
    void* slot_buf;         /* device, capacity * record_bytes */
    void* workspace;        /* device, workspace_bytes from ft_cache_required_sizes;
                               holds the slot tables; contents are owned by the cache */
    const void* shared_experts; /* device, L records (always-resident shared expert,
                               weight 1, [JUHE "先纠正一个容易混淆的模型"]), or NULL */
    ft_split split;
    int32_t format;         /* FT_FORMAT_NVFP4 (0) or FT_FORMAT_MXFP4 of host_pool and
                               shared_experts */
} ft_cache_desc;

/* Bytes of one expert record (padded), for hidden H and intermediate I (NVFP4, and
 * for a given format). */
ft_status ft_record_bytes(int32_t H, int32_t I, size_t* bytes);
ft_status ft_record_bytes_format(int32_t format, int32_t H, int32_t I, size_t* bytes);

/* Record bytes and device workspace bytes needed by a descriptor (host pointers in
 * it are ignored).  The workspace holds the slot tables ([JUHE "生成阶段"]:
 * slot_for_id, id_of_slot, usage), the per-call route and work lists, the h
 * activations and, when T_max > 0, the prefill buffers. */
ft_status ft_cache_required_sizes(const ft_cache_desc* d, size_t* record_bytes,
                                  size_t* workspace_bytes);

/* Create a cache over caller-owned memory.  Synchronous.  The cache starts cold
 * (every slot free, tick 0; [EXPLAINER §7.3]).  Errors: FT_ERR_ARG (sizes, NULL
 * pointers, misaligned buffers), FT_ERR_UNPINNED (host_pool not page-locked),
 * FT_ERR_CUDA. */
ft_status ft_cache_create(const ft_cache_desc* d, ft_cache** out);
void      ft_cache_destroy(ft_cache* c);

/* Safe-point rebuild ([EXPLAINER §7.2]; [JUHE "显存还要在专家缓存和 KV Cache 之间
 * 动态分配"]): synchronises `stream` and the internal copy stream, switches to
 * new_capacity slots in new_slot_buf (may equal the old buffer), empties every
 * table and keeps the host pool; the tick keeps counting.  Errors: FT_ERR_ARG
 * (new_capacity outside [1, capacity_max] or NULL buffer), FT_ERR_STATE (stream is
 * being captured), FT_ERR_CUDA. */
ft_status ft_cache_resize(ft_cache* c, int32_t new_capacity, void* new_slot_buf,
                          void* stream);

/* Replace the miss split used by later calls.  FT_ERR_ARG on a bad mode/f_q16. */
ft_status ft_set_split(ft_cache* c, ft_split s);

/* f = min(1, B_P / B_H) as Q16 ([EXPLAINER §6.5]), floor(f*65536 + 0.5); returns 0
 * when either bandwidth is <= 0. */
uint32_t  ft_split_from_bandwidth(double B_P, double B_H);
/* f = p_ov / (p_ov + c_ov) as Q16 ([BWRATIO "实测版本"]); 0 on invalid input. */
uint32_t  ft_split_from_overlap(double p_ov, double c_ov);

/* One routed-MoE layer of decode ([EXPLAINER §6.1-6.8, §8.2]; [BWRATIO "代码全链路"
 * §2]; [JUHE "生成阶段"]), fully on the device, in stream order:
 *   1. flat = layer*E + id for every route; dedupe across the batch (ascending);
 *   2. hit iff slot_for_id[flat] >= 0; |H| hits, m unique misses;
 *   3. q from the split, capped at C - |H|;
 *   4. the q LRU slots not touched by this call (free slots first, ascending, then
 *      ascending (usage, slot)) take the first q misses in ascending flat id;
 *      evicted ids are unmapped; every touched slot gets usage = tick (one tick per
 *      call, touched slots ordered by slot index);
 *   5. the q fills are read from the pinned pool once, written into their slots and
 *      computed on the way (load-through over the host link);
 *   6. NVFP4 SwiGLU per unique GPU expert (hits + fills, + the shared expert);
 *   7. y[b] = sum_j w[b,j] * o_(b,j) over GPU routes, + shared(x_b); the terms are
 *      fp32 adds in no fixed order, so y can differ between calls in the last bits.
 * Arguments:
 *   x          device bf16 [B, H]
 *   topk_ids   device int32 [B, k], local expert ids; an id outside [0, E) masks the
 *              route (neither hit, miss nor deferred) and sets FT_DEV_BAD_ID
 *   topk_w     device fp32 [B, k] gates
 *   y          device fp32 [B, H], overwritten (GPU partial: routes on the host share
 *              contribute 0)
 *   deferred   device int32 [B, k]: flat id of each route left to the host share
 *              ([EXPLAINER §6.2] set C), else -1
 *   route_slot device int32 [B, k] or NULL: slot used by each route, else -1
 *   counters   device int32 [4] or NULL: n_hit (|H|), m, q, deferred routes
 * Errors (host-side, nothing launched): FT_ERR_ARG for layer outside [0, L),
 * B outside [1, B_max], k outside [1, k_max] or NULL x/ids/w/y/deferred. */
ft_status ft_moe_decode(ft_cache* c, int32_t layer, const void* x, const int32_t* topk_ids,
                        const float* topk_w, int32_t B, int32_t k, float* y,
                        int32_t* deferred, int32_t* route_slot, int32_t* counters,
                        void* stream);

/* ft_moe_decode with no allocation and no per-call workspace: the same layer call
 * (same arguments, same results, same cache state) whose per-call scratch lives in
 * a static 8 MiB device array built into the library instead of the workspace.
 * The paper has no counterpart; it serves callers that cannot allocate device
 * memory (a host framework that owns all device memory through its own pool, or a
 * serving loop that must never enter the CUDA allocator).  The array's device
 * address is looked up on the first call made on each device, so make that first
 * call before any stream capture.  Every call shares the array: calls that
 * overlap on the GPU race and must be serialised by the caller.  Errors: those of
 * ft_moe_decode, and FT_ERR_ARG when B, k, H and I need more than 8 MiB of scratch:
 * (B*k + B) * I * 8 bytes of h words and (H / rows) * 8 bytes of tile flags, each
 * region rounded up to 256 bytes, plus 256 bytes of grid state (rows = 64 at the
 * benchmark shapes). */
ft_status ft_moe_decode_static(ft_cache* c, int32_t layer, const void* x,
                               const int32_t* topk_ids, const float* topk_w, int32_t B,
                               int32_t k, float* y, int32_t* deferred, int32_t* route_slot,
                               int32_t* counters, void* stream);

/* Prefill of one layer over a T-token chunk ([EXPLAINER §4.1-4.3]; [JUHE "Prefill 为什么
 * 不能也按需加载"]).  With FT_PREFILL_DOUBLE_BUFFER and capacity >= 2E the layer's
 * experts sit in buffer (layer mod 2) = slots [(layer%2)*E, +E) and, while this layer
 * computes, every expert of layer+1 streams into the other buffer on the internal copy
 * stream.  Without the flag and with capacity >= E only buffer 0 is used and each
 * layer is loaded before it computes.  Otherwise (two layers do not fit for the double
 * buffer, one does not fit for the single one) or with FT_PREFILL_ON_DEMAND, the call
 * falls back to loading on demand: the layer's routed union (experts with at least one
 * valid route, ascending id) goes through the global LRU like decode misses with every
 * miss filled, in groups of at most C experts (one tick per group, the first group
 * ticks even for an empty union); each group's missing records are streamed from the
 * pinned pool into their victim slots by the GPU (in batches on the cache's copy
 * stream, each batch computed beside the next one's stream-in) and the group is
 * computed before the next one may evict it.  What is resident afterwards is decode's cache.  Activations and h are NVFP4 (unit
 * tensor scale, E4M3 per 16); the two grouped GEMMs run on tcgen05 block-scaled
 * FP4 tensor cores; y[t] = sum_j w[t,j] * o_(t,j) in order j.
 *   x         device bf16 [T, H];  topk_ids device int32 [T, k];  topk_w device fp32 [T, k]
 *   y         device fp32 [T, H], overwritten
 *   debug_h   device uint8 or NULL: per route r = t*k + j, I/2 packed h codes followed
 *             (after all T*k rows) by [T*k, I/16] h scales.  With FT_PREFILL_DEBUG_X
 *             in flags, the same buffer continues with the quantised activations as
 *             the GEMM reads them: int32 [T*k] sorted row of each route (-1: masked
 *             route), then [T*k, H/2] packed x codes and [T*k, H/16] x scales in
 *             sorted-row order (rows past the last valid route are unspecified).
 *             Total bytes: T*k*(I/2 + I/16 + 4 + H/2 + H/16).
 * Calls for one chunk go layer 0, 1, ..., L-1 on the same stream.
 * Errors (host-side, nothing launched): FT_ERR_STATE when the cache was created with
 * T_max = 0; FT_ERR_ARG for H or I not multiples of 256, layer outside [0, L), T
 * outside [1, T_max], k outside [1, k_max], NULL x/ids/w/y, x or y not 16-byte
 * aligned, or an unknown flag.  Route ids outside [0, E), or repeating an id of their
 * own token, mask the route and set FT_DEV_BAD_ID. */
#define FT_PREFILL_DOUBLE_BUFFER 1
#define FT_PREFILL_DEBUG_X       2
#define FT_PREFILL_ON_DEMAND     4
ft_status ft_moe_prefill_layer(ft_cache* c, int32_t layer, const void* x,
                               const int32_t* topk_ids, const float* topk_w, int32_t T,
                               int32_t k, float* y, int32_t flags, void* debug_h,
                               void* stream);

/* Copy the tables to host arrays (synchronises the cache's streams):
 * slot_for_id [L*E], id_of_slot [C], usage [C] (-1 = never used since the last
 * resize), tick.  Any output may be NULL. */
ft_status ft_cache_snapshot(ft_cache* c, int32_t* slot_for_id, int32_t* id_of_slot,
                            int64_t* usage, int64_t* tick);

/* Load the tables from host arrays, the inverse of ft_cache_snapshot (for replaying a
 * run from a saved point; the slot contents are not saved, so every occupied slot
 * must already hold its expert's record, e.g. the buffer the snapshot was taken
 * over).  Synchronous safe-point call like ft_cache_resize: synchronises `stream`
 * and the copy stream, then writes slot_for_id [L*E], id_of_slot [C], usage [C] and
 * the tick, and rebuilds the LRU order (free slots ascending, then ascending
 * (usage, slot)).  The arrays must be consistent: id_of_slot[s] in [-1, L*E),
 * slot_for_id[f] in [-1, C), slot_for_id[id_of_slot[s]] == s for every occupied s
 * and id_of_slot[slot_for_id[f]] == f for every mapped f, usage -1 exactly on free
 * slots and in [0, tick] elsewhere.  Errors: FT_ERR_ARG (NULL array, inconsistent
 * tables), FT_ERR_STATE (stream is being captured), FT_ERR_CUDA. */
ft_status ft_cache_restore(ft_cache* c, const int32_t* slot_for_id, const int32_t* id_of_slot,
                           const int64_t* usage, int64_t tick, void* stream);

/* Per-call stats ring (device).  When set, every decode call (ft_moe_decode,
 * ft_moe_decode_static) appends one record from its commit step: the call's tick,
 * layer, |H|, m, q, deferred routes, the number of GPU experts computed (hits +
 * fills + the shared expert) and the GPU's %globaltimer at the commit (ns).
 * ring: device memory of 16 + capacity * sizeof(ft_trace_rec) bytes, 16-byte
 * aligned, zeroed by the caller: uint64 count (records ever written), 8 bytes
 * reserved, then the records; record i lands at index i mod capacity.  ring NULL or
 * capacity 0 switches the ring off.  Only later calls see the change. */
typedef struct {
    int64_t tick;
    int32_t layer, n_hit, m, q, n_def_routes, n_units;
    int64_t t_commit_ns;
} ft_trace_rec;
ft_status ft_cache_set_trace(ft_cache* c, void* ring, int32_t capacity);

/* Current slot count. */
ft_status ft_cache_capacity(const ft_cache* c, int32_t* capacity);

/* Read and clear the device status word (FT_DEV_* bits).  Synchronises. */
ft_status ft_cache_status(ft_cache* c, int32_t* device_status);

/* Diagnostic of the failure path (no counterpart on the pages): one GPU thread runs
 * each kind of bounded wait the decode kernel uses against a condition nothing will
 * satisfy (a counter nobody raises, a tagged word nobody writes, read once with an
 * acquire and once in a batch, an mbarrier nobody arrives on).  Every wait must give
 * up after its one-second bound instead of hanging; *expired gets bit i set when wait
 * i did, so a healthy build returns 0xF.  The kernel exits normally and the context
 * stays usable.  Takes about 4 s; synchronises the device; needs no cache.
 * Errors: FT_ERR_ARG for a NULL expired, FT_ERR_CUDA when the launch fails. */
ft_status ft_check_bounded_waits(uint32_t* expired);

/* Quantise n experts to NVFP4 records on the device ([EXPLAINER §8.4] layout; the
 * quantiser of the record format above, fp32 IEEE steps):
 *   s_t = amax(W)/2688; block scale = E4M3_RNE((amax16/6)/s_t);
 *   code = E2M1_RNE_sat(w / (scale*s_t)); a zero scale gives a zero block.
 *   w_gu device fp32 [n, 2I, H];  w_d device fp32 [n, H, I];
 *   records device uint8 [n, ft_record_bytes(H, I)]. */
ft_status ft_quantize_experts(const float* w_gu, const float* w_d, int32_t n, int32_t H,
                              int32_t I, void* records, void* stream);
/* The same for MXFP4 records (the conversion rule of the microscaling format, fp32 IEEE
 * steps): shared = floor(log2(amax32)) - 2 clamped to [-127, 127] (amax 0: -127);
 * scale code = shared + 127; code = E2M1_RNE_sat(w * 2^-shared); tensor scales 1.0.
 * records device uint8 [n, ft_record_bytes_format(FT_FORMAT_MXFP4, H, I)]. */
ft_status ft_quantize_experts_mx(const float* w_gu, const float* w_d, int32_t n, int32_t H,
                                 int32_t I, void* records, void* stream);

/* Page-locked, device-mapped host memory for the pool ([EXPLAINER §7.3]: pin the
 * pool; the caller fills it). */
ft_status ft_pinned_alloc(size_t bytes, void** out);
ft_status ft_pinned_free(void* p);

/* Effective pinned-host -> device bandwidth in GB/s ([EXPLAINER §6.3] B_P; [QIITA §7]):
 * best of `reps` timed cudaMemcpyAsync of `bytes` from `pinned` to `dev`. */
ft_status ft_measure_h2d(const void* pinned, void* dev, size_t bytes, int32_t reps,
                         double* gbps);

/* Per-kernel device time accumulated while profiling is on (CUDA events around
 * each launch on the launching stream).  kind: 0 decode layer kernel, 1 prefill
 * GEMM1, 2 prefill GEMM2, 3 prefill other kernels, 4 prefill layer copies (on the
 * cache's copy stream).  kinds: bit mask, bit i times launches of kind i (0: off,
 * FT_PROF_ALL: every kind).  Timing only the copies (kinds = 1 << 4) records events
 * on the copy stream alone and leaves the compute stream's launches untouched. */
#define FT_PROF_KINDS 5
#define FT_PROF_ALL ((1 << FT_PROF_KINDS) - 1)
ft_status ft_profile_enable(ft_cache* c, int32_t kinds);
ft_status ft_profile_read(ft_cache* c, double* total_ms /*[FT_PROF_KINDS]*/,
                          int64_t* launches /*[FT_PROF_KINDS]*/);

/* ---- The host share of decode ([EXPLAINER §8.3]; [BWRATIO "代码全链路" §2]; [JUHE
 * "为什么可以直接相加？"]).
 * A host branch is a persistent pool of n_threads worker threads, each pinned to one
 * CPU core, that computes routes left to the host (deferred >= 0) straight from the
 * pinned pool: the same SwiGLU expert on the records' codes and scales, dequantised
 * inside the GEMV (NEON on aarch64), with fp32 products and sums:
 *   y[b] += w[b,j] * Expert_{deferred[b,j]}(x[b]) over the host routes, experts in
 *   ascending flat id.
 * Attached to a cache (ft_cache_set_host_branch), every decode call hands its host
 * share to the branch right after its decision: the decode kernel writes the call's
 * deferred ids, gates and x into the branch's mailbox (pinned, device-mapped) and
 * raises a flag; worker 0 sees it, the workers compute the host partial into the
 * mailbox while the GPU computes its own share, and a join kernel, launched on the
 * call's stream right after the decode kernel, waits for the branch (bounded: one
 * second, then FT_DEV_TIMEOUT) and adds the host partial into y.  y then holds the
 * whole layer output y_gpu + y_cpu; a call with no host routes joins nothing.
 * Both calls stay asynchronous and capturable; the branch's workers spin while calls
 * arrive and back off when idle. */
typedef struct ft_host_branch ft_host_branch;
typedef struct {
    int32_t L, E, H, I, k_max, B_max, format;   /* as the cache's descriptor */
    const void* host_pool;   /* pinned pool (the cache's), L*E records */
    int32_t n_threads;       /* workers, >= 1 */
    const int32_t* cpus;     /* n_threads CPU ids to pin the workers to, or NULL: the
                                first n_threads CPUs this process may run on */
    void* mailbox;           /* pinned (ft_pinned_alloc), 256-byte aligned,
                                ft_host_mailbox_bytes(H, k_max, B_max) bytes; NULL:
                                the branch only serves ft_host_moe */
} ft_host_desc;
/* Bytes of a mailbox for hidden H, k_max, B_max.  FT_ERR_ARG on bad sizes. */
ft_status ft_host_mailbox_bytes(int32_t H, int32_t k_max, int32_t B_max, size_t* bytes);
/* Start a branch (threads created and pinned).  FT_ERR_ARG on bad fields. */
ft_status ft_host_branch_create(const ft_host_desc* d, ft_host_branch** out);
/* Stop and join the workers.  Detach the branch from every cache first. */
void      ft_host_branch_destroy(ft_host_branch* hb);
/* The host share of one call, computed now by the workers (synchronous; host memory):
 *   x host bf16 [B, H]; deferred host int32 [B, k] flat ids (l*E + e) or -1;
 *   w host fp32 [B, k]; y host fp32 [B, H], overwritten with the host partial.
 * Not to be called while decode calls on an attached cache are in flight.
 * Errors: FT_ERR_ARG (NULL pointer, B outside [1, B_max], k outside [1, k_max]). */
ft_status ft_host_moe(ft_host_branch* hb, const void* x, const int32_t* deferred, const float* w,
                      int32_t B, int32_t k, float* y);
/* Jobs run by the branch (all, and those published by decode kernels). */
ft_status ft_host_branch_stats(const ft_host_branch* hb, int64_t* jobs, int64_t* mailbox_jobs);
/* Attach hb (or detach with NULL): later decode calls of c hand their host share to
 * it and add its partial into y.  hb must describe c's shape, format and pool, with
 * B_max and k_max at least the cache's, and have a mailbox.  Synchronises the cache's
 * streams.  Errors: FT_ERR_ARG (mismatch), FT_ERR_CUDA. */
ft_status ft_cache_set_host_branch(ft_cache* c, ft_host_branch* hb);

/* ---- Bandwidth profile ([EXPLAINER §6.3]; [BWRATIO "第一层带宽比", "实测版本"];
 * [QIITA §7]): the two real miss paths over the same n_records records of the pool
 * (flat ids 0 .. n_records-1), in record bytes per second:
 *   pcie_gbs      the GPU fill path alone: the records gathered from the pinned pool
 *                 into slots 0 .. n_records-1 by the GPU's gather kernel;
 *   cpu_gbs       the host branch alone: its workers computing one token through
 *                 every record (ft_host_moe's GEMV);
 *   pcie_ov_gbs, cpu_ov_gbs   both started together, each over its own duration.
 * recommend = ft_recommend_backend(cpu_gbs, pcie_gbs); f_q16 =
 * ft_split_from_overlap(pcie_ov_gbs, cpu_ov_gbs).  A safe-point call: synchronises,
 * and leaves the cache empty (like ft_cache_resize to the same capacity); allocates
 * and frees 8 * n_records + 16 bytes of device memory.  Errors: FT_ERR_ARG
 * (n_records outside [1, min(C, L*E)], NULL pointers, a branch of another pool or
 * shape), FT_ERR_STATE (capturing), FT_ERR_CUDA. */
#define FT_BACKEND_OFFLOAD 0
#define FT_BACKEND_HYBRID  1
typedef struct {
    double pcie_gbs, cpu_gbs, pcie_ov_gbs, cpu_ov_gbs;
    int32_t recommend;
    uint32_t f_q16;
    int32_t n_records;
} ft_bw_profile;
ft_status ft_profile_bandwidth(ft_cache* c, ft_host_branch* hb, int32_t n_records, void* stream,
                               ft_bw_profile* out);
/* [BWRATIO "第一层带宽比"]: FT_BACKEND_HYBRID when the CPU expert path is more than
 * twice as fast as the fill path (cpu_gbs > 2 * pcie_gbs), else FT_BACKEND_OFFLOAD. */
int32_t   ft_recommend_backend(double cpu_gbs, double pcie_gbs);

const char* ft_status_string(ft_status s);
/* Message of the last failed call on c (static storage), or "" */
const char* ft_last_error(const ft_cache* c);

#ifdef __cplusplus
}
#endif
#endif /* FT_H */
