/*
 * pe.h -- C ABI of libpe, a single-GPU paged MoE layer for GB300 (sm_103a).
 *
 * What it computes ("Paged Experts", SGLang docs):
 *   "The K-slot table and the host store": each MoE layer keeps K of its E
 *   routed experts in a K-slot table in GPU memory and all E experts in a
 *   page-locked host store whose rows have exactly the slot layout.
 *   "A step: waves, page-in, merge": every forward step of a layer routes the
 *   tokens (softmax over E, top-k, renormalise), splits the distinct routed
 *   experts into waves of at most K with the resident ones first, makes each
 *   wave resident by evicting the least recently used experts outside it,
 *   copies the missing experts from the host store into their slots, remaps
 *   routed ids to slots, runs the SiLU-gated expert MLP of every routed
 *   (token, expert) entry times its router weight into one merged buffer, and
 *   finally sums each token's top-k entries.
 *   "Captured decode": planning and page-in run on the GPU from device-side
 *   counts, so a forward call never synchronises with the host and can be
 *   captured in a CUDA graph; captured and uncaptured calls share one LRU
 *   state.
 *
 * Conventions for every call:
 *   - Plain C types only.  "device pointer" = memory of the configured CUDA
 *     device; "host pointer" = ordinary CPU memory.
 *   - Return value: PE_OK or an error code; the message of the last error of
 *     a handle is available from pe_last_error().  No call throws or aborts.
 *   - A handle is used from one host thread at a time, and its forward calls
 *     must be ordered on one CUDA stream (they share one workspace).
 *   - Errors detected on the GPU (NaN logits, routed experts never loaded,
 *     ids out of range) do not fail the asynchronous call; they set bits of a
 *     device error word that pe_stats() returns.
 */
#ifndef PE_H_
#define PE_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pe_status {
    PE_OK = 0,
    PE_ERR_INVALID = 1,           /* bad configuration or argument           */
    PE_ERR_UNSUPPORTED_DTYPE = 2, /* expert format not among pe_dtype        */
    PE_ERR_HOST_ALLOC = 3,        /* host store could not be pinned          */
    PE_ERR_CUDA = 4,              /* a CUDA runtime call failed              */
    PE_ERR_RANGE = 5,             /* layer/expert/slot/token count too large */
    PE_ERR_ARENA = 6              /* device arena missing, misaligned, small */
} pe_status;

/* Expert storage formats ("Paged Experts", "Supported Configurations and
 * Limitations": unquantised, block-quantised FP8 with 128x128 blocks, and
 * GPTQ int4; "SGLang Paged Experts: corré MoE más grandes que tu VRAM",
 * "¿Qué es la paginación de expertos…?": MXFP4 and NVFP4 as well; other
 * formats are rejected at creation).  Activations stay bf16 in every format. */
typedef enum pe_dtype {
    PE_BF16 = 0,          /* bf16 weights                                    */
    PE_FP8_BLOCK128 = 1,  /* E4M3 weights, one fp32 scale per 128x128 block  */
    PE_INT4_GPTQ = 2,     /* GPTQ int4: 4-bit codes, zero point 8, one fp16
                             scale per output row and group of 128 inputs    */
    PE_MXFP4 = 3,         /* E2M1 codes, one E8M0 scale per row and 32 inputs*/
    PE_NVFP4 = 4          /* E2M1 codes, one E4M3 scale per row and 16
                             inputs, times one fp32 scale per tensor         */
} pe_dtype;

/* Device error word bits (read through pe_stats). */
#define PE_DEVERR_NAN_LOGIT  0x1u /* a router logit was NaN (routed as -inf) */
#define PE_DEVERR_NOT_LOADED 0x2u /* a planned expert was never loaded       */
#define PE_DEVERR_PLAN       0x4u /* internal plan check failed              */
#define PE_DEVERR_TIMEOUT    0x8u /* a bounded wait inside a kernel gave up   */

typedef struct pe_config {
    int32_t num_layers;   /* L, MoE layers sharing one host store         */
    int32_t num_experts;  /* E, routed experts per layer (1..1024)        */
    int32_t top_k;        /* experts per token (1..min(E, 32))            */
    int32_t num_slots;    /* K, resident experts per layer (top_k..E)     */
    int32_t hidden;       /* H, model width (multiple of 8; of 128 for FP8, int4, FP4)*/
    int32_t intermediate; /* I, expert width (multiple of 8; of 128 for FP8, int4;
                             of the 32- or 16-input block for MXFP4, NVFP4)    */
    int32_t dtype;        /* pe_dtype                                     */
    int32_t max_tokens;   /* largest num_tokens a forward call may pass   */
    int32_t device;       /* CUDA device ordinal                          */
} pe_config;

/* Byte layout of one expert row; a host-store row and a slot are identical.
 * bf16: w13 = [2I, H] (rows 0..I-1 gate projection, I..2I-1 up projection),
 *       w2 = [H, I] (down projection), both row-major bf16; no scales.
 * FP8:  w13 and w2 as E4M3 codes (one byte each, same shapes), s13 =
 *       [ceil(2I/128), ceil(H/128)] and s2 = [ceil(H/128), ceil(I/128)]
 *       row-major fp32 block scales.
 * int4: w13 = [2I, H/2] and w2 = [H, I/2] bytes, byte j of a row holding
 *       input 2j in its low nibble and 2j+1 in its high nibble; the weight
 *       is (code - 8) * scale with s13 = [2I, H/128] and s2 = [H, I/128]
 *       row-major fp16 scales (one per output row and 128 inputs).  A GPTQ
 *       checkpoint (8 codes per int32 along the input, scales [K/128, N])
 *       maps to this by a transpose of both.
 * MXFP4 / NVFP4: E2M1 codes packed as for int4, with I padded to Ip, the
 *       next multiple of 128 (zero codes and scales): w13 = [2Ip, H/2]
 *       (gate rows 0.., up rows Ip..), w2 = [H, Ip/2]; s13 = [2Ip, H/B] and
 *       s2 = [H, Ip/B] one-byte block scales, B = 32 (MXFP4, E8M0) or 16
 *       (NVFP4, E4M3); for NVFP4 each grid follows a 16-byte header whose
 *       first 4 bytes are the tensor's fp32 scale.  pe_load_host_expert takes
 *       the logical (unpadded) tensors and writes this layout.
 * Offsets are 128-byte aligned. */
typedef struct pe_row_layout {
    uint64_t w13_offset, w13_bytes;
    uint64_t s13_offset, s13_bytes;  /* 0 bytes for bf16 */
    uint64_t w2_offset, w2_bytes;
    uint64_t s2_offset, s2_bytes;    /* 0 bytes for bf16 */
    uint64_t payload_bytes;          /* w13+s13+w2+s2: the expert's size  */
    uint64_t row_stride;             /* distance between rows (256-aligned)*/
} pe_row_layout;

/* Cumulative per-layer counters since creation (or the sum over layers). */
typedef struct pe_stats_t {
    uint64_t steps;       /* forward calls                                  */
    uint64_t waves;       /* waves planned                                  */
    uint64_t entries;     /* routed (token, expert) entries                 */
    uint64_t distinct;    /* distinct experts routed, summed over steps     */
    uint64_t hits;        /* distinct experts already resident              */
    uint64_t page_ins;    /* experts copied from the host store             */
    uint64_t cold_fills;  /* page-ins into a slot that was empty            */
    uint64_t bytes_paged; /* page_ins * payload bytes                       */
    uint32_t error_word;  /* PE_DEVERR_* bits, sticky                       */
    uint32_t reserved;
} pe_stats_t;

/* The last step's plan of a layer, copied to caller-owned host arrays.
 * max_waves = pe_max_waves(cfg, num_tokens). */
typedef struct pe_plan_view {
    int32_t* plan_expert; /* [max_waves][K]: experts copied in, per wave    */
    int32_t* plan_slot;   /* [max_waves][K]: their slots                    */
    int32_t* plan_count;  /* [max_waves]: experts copied in each wave       */
    int32_t* topk_id;     /* [T*top_k]: routed ids, descending logit        */
    float* topk_w;        /* [T*top_k]: renormalised router weights         */
    int32_t* entry_slot;  /* [T*top_k]: slot of each entry in its wave      */
    int32_t* entry_wave;  /* [T*top_k]: wave holding each entry's expert    */
    int32_t num_waves;    /* out: waves the step used                       */
} pe_plan_view;

/* Per-kernel device time recorded while profiling is on. */
#define PE_PROF_KINDS 12
typedef struct pe_profile_t {
    const char* name[PE_PROF_KINDS]; /* kernel family; NULL if unused        */
    uint64_t launches[PE_PROF_KINDS];
    double total_ms[PE_PROF_KINDS];  /* CUDA-event time on the call's stream */
} pe_profile_t;

typedef struct pe_handle pe_handle;

/* Device bytes the caller must provide to pe_create for this config: the
 * L*K slot table, per-layer LRU state and plans, and the forward workspace
 * for up to max_tokens tokens (with the tensor-core prefill path and steps
 * of two or more waves, also K staging rows after the slot table, where a
 * later wave's page-in lands while its slot is still in use).  Returns 0 for
 * an invalid config.  Pure. */
size_t pe_required_device_bytes(const pe_config* cfg);

/* Slot count for a device-memory budget.  "Paged Experts" (SGLang docs),
 * "Choosing K": the slot table competes with the rest of GPU memory, and one
 * resident slot costs expert_bytes x num_moe_layers, so K is what the budget
 * left for it allows.  Returns the largest K, top_k <= K <= num_experts, for
 * which pe_required_device_bytes(cfg with num_slots = K) <= budget_bytes
 * (the whole arena, slot table and workspace, is counted); 0 if even
 * K = top_k does not fit or the config is invalid for every K.
 * cfg->num_slots is ignored.  Pure. */
int32_t pe_slots_for_budget(const pe_config* cfg, size_t budget_bytes);

/* Row layout for a config (see pe_row_layout).  Pure. */
pe_status pe_get_row_layout(const pe_config* cfg, pe_row_layout* out);

/* Upper bound on the waves one step with num_tokens tokens can need:
 * 1 when num_tokens*top_k <= K, else ceil(min(E, num_tokens*top_k) / K).
 * Derived from shapes only, so it needs no device data.  Pure. */
int32_t pe_max_waves(const pe_config* cfg, int32_t num_tokens);

/* Create a paged layer stack.
 *   dev_arena:   caller-owned device memory, 256-byte aligned, at least
 *                pe_required_device_bytes(cfg) bytes; the library keeps a
 *                pointer into it until pe_destroy and never frees it.  The
 *                library allocates no device memory itself.
 *   The library allocates and owns the page-locked host store
 *   (L*E*row_stride bytes, mapped into the device address space).
 *   All slots start empty.  Synchronises the device once.
 * Errors: PE_ERR_INVALID (top_k > K, K > E, sizes out of range, bad device),
 *   PE_ERR_UNSUPPORTED_DTYPE, PE_ERR_ARENA, PE_ERR_HOST_ALLOC, PE_ERR_CUDA. */
pe_status pe_create(const pe_config* cfg, void* dev_arena, size_t arena_bytes, pe_handle** out);

/* Like pe_create, but the new handle reads the host store of `store_owner`
 * (a handle from pe_create or pe_create_external; same L, E, H, I and dtype
 * required; K and max_tokens may differ).  The owner must outlive the new
 * handle.  Used to run the same experts with another K, e.g. K=E as the
 * unpaged reference. */
pe_status pe_create_shared(const pe_config* cfg, void* dev_arena, size_t arena_bytes,
                           pe_handle* store_owner, pe_handle** out);

/* Like pe_create, but the host store is caller-owned memory: host_store must
 * be 4096-byte aligned, hold at least L*E*row_stride bytes (row_stride from
 * pe_get_row_layout) and stay valid until pe_destroy.  It is how several
 * replica processes on one host read ONE copy of the experts ("Paged
 * Experts", "Supported Configurations and Limitations": every expert of every
 * layer has to be page-locked in host memory, so N private copies would need
 * N times the host memory): one process maps a shared region (a file under
 * /dev/shm, say), fills it through a handle created with filled = 0 and
 * pe_load_host_expert, and every replica, that one included, creates its
 * handle on the same mapping with filled = 1, which marks every expert loaded.
 * The library registers the memory (cudaHostRegister, mapped and portable)
 * while any handle of this process uses it (handles on the same store share
 * one registration, released with the last of them in pe_destroy); it never
 * frees it.  A handle with filled = 1 only reads the store.
 * Errors: as pe_create; PE_ERR_INVALID for a NULL, misaligned or too small
 *   store (checked before any CUDA call); PE_ERR_HOST_ALLOC if the
 *   registration fails. */
pe_status pe_create_external(const pe_config* cfg, void* dev_arena, size_t arena_bytes, void* host_store,
                             size_t host_store_bytes, int32_t filled, pe_handle** out);

/* Copy one expert into its host-store row (a synchronous host memcpy),
 * through the handle that created or registered the store.
 *   w13, w2: host pointers in the row layout's formats (bf16 bits, E4M3
 *   codes or packed 4-bit codes); s13, s2: the scales, fp32 for FP8 and fp16
 *   for int4, NULL for bf16.  MXFP4 / NVFP4 take their logical shapes
 *   (w13 [2I, H/2], w2 [H, I/2] bytes; scales [2I, H/B] and [H, I/B] bytes,
 *   B = 32 or 16), and for NVFP4 each scale pointer starts with a 16-byte
 *   header holding the tensor's fp32 scale (then 12 ignored bytes); the
 *   library writes them into the padded row layout, zeros included.
 *   Marks the expert loaded; a later forward that routes to an expert that
 *   was never loaded sets PE_DEVERR_NOT_LOADED.  Loading an expert that is
 *   currently resident does not refresh its slot: load before forwarding, or
 *   call pe_reset_residency afterwards.
 * Errors: PE_ERR_RANGE (layer/expert), PE_ERR_INVALID (NULL or stray
 *   scale pointers), PE_ERR_CUDA. */
pe_status pe_load_host_expert(pe_handle* h, int32_t layer, int32_t expert, const void* w13,
                              const void* w2, const void* s13, const void* s2);

/* Host pointer to an expert's row in the host store (for inspection). */
void* pe_host_row(pe_handle* h, int32_t layer, int32_t expert);

/* One forward step of MoE layer `layer`, asynchronous on `stream`
 * (a cudaStream_t; NULL = the legacy default stream).
 *   hidden:        device, bf16 [num_tokens, H] row-major
 *   router_logits: device, fp32 [num_tokens, E] row-major
 *   out:           device, bf16 [num_tokens, H]; written, may not alias hidden
 *   num_tokens:    1..max_tokens (0 is a no-op)
 * Launches only kernels on `stream` (route+plan, page-in, expert MLP,
 * merge/top-k sum); makes no host synchronisation and no allocation, so it
 * may be captured in a CUDA graph.  The output does not depend on K or on
 * how the experts were split into waves: it is bit-identical to the same
 * call on a handle with K = E.
 * Errors (synchronous): PE_ERR_RANGE, PE_ERR_INVALID (NULL pointers),
 *   PE_ERR_CUDA (launch failure). */
pe_status pe_forward(pe_handle* h, int32_t layer, const void* hidden, const float* router_logits,
                     void* out, int32_t num_tokens, void* stream);

/* Counters of one layer (layer >= 0) or summed over all layers (layer = -1).
 * Synchronises the device first; not capturable. */
pe_status pe_stats(pe_handle* h, int32_t layer, pe_stats_t* out);

/* Copy the last step's plan of `layer` (called with that step's num_tokens)
 * into caller-owned host arrays.  Synchronises the device. */
pe_status pe_read_plan(pe_handle* h, int32_t layer, int32_t num_tokens, pe_plan_view* out);

/* Copy a layer's residency state to host arrays: slot_expert [K] (-1 =
 * empty), slot_tick [K], expert_slot [E] (-1 = not resident), clock.
 * Any pointer may be NULL.  Synchronises the device. */
pe_status pe_read_residency(pe_handle* h, int32_t layer, int32_t* slot_expert, uint32_t* slot_tick,
                            int32_t* expert_slot, uint32_t* clock);

/* Copy `bytes` (<= row_stride) of slot `slot` of `layer` to host memory.
 * Synchronises the device. */
pe_status pe_read_slot(pe_handle* h, int32_t layer, int32_t slot, void* host_dst, size_t bytes);

/* Empty every slot of every layer and zero the clocks (counters and the
 * error word are kept), asynchronously on `stream`. */
pe_status pe_reset_residency(pe_handle* h, void* stream);

/* Self-test of failure detection, without a GPU fault.  Every wait inside
 * the kernels is bounded: on running out it records PE_DEVERR_TIMEOUT in an
 * error word and returns, so the context stays usable.  This runs, on the
 * current device, each kind of wait the kernels use on a condition that
 * never becomes true, with `poll_limit` polls (about 0.1-1 us each):
 *   out3[0]  the prefill step's counter wait (bit 31 set if it did not also
 *            raise the step's abort word, which must end a second wait at once);
 *   out3[1]  an mbarrier wait (the tensor-core pipeline's);
 *   out3[2]  the decode step's phase wait.
 * Each word must read PE_DEVERR_TIMEOUT.  Returns PE_ERR_INVALID for a NULL
 * out3 or a zero limit, PE_ERR_CUDA if a launch failed.  Synchronises the
 * device. */
pe_status pe_selftest_bounded_waits(uint32_t poll_limit, uint32_t* out3);

/* Measure the host link: copy `bytes` of the host store to `dev_dst`
 * (caller-owned device memory) `iters` times with cudaMemcpyAsync and with
 * the page-in kernel's device-side loads, timed with CUDA events on
 * `stream`.  Writes GB/s (1e9 bytes/s) of each.  bytes is clamped to the
 * store size.  Synchronises the stream. */
pe_status pe_probe_host_link(pe_handle* h, void* dev_dst, size_t bytes, int32_t iters, void* stream,
                             double* copy_engine_gbs, double* kernel_gbs);

/* Per-kernel timing: while on, every kernel launch of pe_forward is
 * bracketed by CUDA events on its stream (do not capture while on).
 * pe_profile_read synchronises, fills `out` with the totals since the last
 * pe_profile_enable(h, 1), and keeps profiling on. */
pe_status pe_profile_enable(pe_handle* h, int32_t on);
pe_status pe_profile_read(pe_handle* h, pe_profile_t* out);

/* Scratch held by pe_expert_mlp_noalloc in every GPU that loads libpe. */
#define PE_NOALLOC_SCRATCH_BYTES (1u << 20)

/* One bf16 expert's SiLU-gated MLP that allocates nothing, for callers that
 * cannot allocate device memory where they need it (for example code that
 * may only use the buffers a framework hands it, or a path that must not
 * synchronise the device by calling cudaMalloc).  The pages describe no such
 * call; it has no counterpart there.
 *   out[t] = w2 . (SiLU(w13[0:I] . x[t]) * (w13[I:2I] . x[t]))  for t < num_tokens
 *   w13: device, bf16 [2I, H] (gate rows, then up rows); w2: device, bf16 [H, I];
 *   x, out: device, bf16 [num_tokens, H]; all 16-byte aligned; out may not
 *   alias x.  H <= 2048 and I <= 1024, both multiples of 8.
 * The intermediate h (num_tokens * I fp32) lives in a static device array of
 * PE_NOALLOC_SCRATCH_BYTES; larger requests return PE_ERR_RANGE before any
 * launch.  For num_tokens <= 64 the result equals pe_forward on a one-expert
 * layer (E = K = top_k = 1) with the same weights bit for bit: both run the
 * same GEMV arithmetic.  Above 64 tokens pe_forward switches to its
 * tensor-core path, which rounds h to bf16 and sums in another order, so
 * there the two agree only within bf16 rounding (rel-L2 well under 1e-2).
 * The first call on a device looks up the array's device address with that
 * device current; make that first call before any stream capture.  Every
 * call shares the one array per device: calls whose kernels overlap on the
 * GPU (other streams, other host threads) race on it; order them on one
 * stream.  Asynchronous on `stream`; no host synchronisation.
 * Errors: PE_ERR_INVALID (NULL, misaligned, bad sizes), PE_ERR_RANGE (above
 *   the limits), PE_ERR_CUDA; the message is in pe_last_error(NULL). */
pe_status pe_expert_mlp_noalloc(const void* w13, const void* w2, const void* x, void* out,
                                int32_t num_tokens, int32_t hidden, int32_t intermediate, void* stream);

/* Frees the host store (if owned) and the handle; never the arena. */
void pe_destroy(pe_handle* h);

/* Message of the handle's last error ("" if none); pe_last_error(NULL)
 * returns the last error of a failed pe_create, or of a failed call that
 * takes no handle, in this thread. */
const char* pe_last_error(pe_handle* h);

#ifdef __cplusplus
}
#endif

#endif /* PE_H_ */
