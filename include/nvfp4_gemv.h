/*
 * nvfp4_gemv.h: C ABI of the NVFP4 (nvfp4/g16) weight-only GEMV library for GB300 (sm_103a).
 *
 * Operation (all entry points):
 *
 *     y[m, n] = g * sum_k E2M1(q[n, k]) * E4M3(s[n, k / 16]) * x[m, k]
 *
 * The weight is NVFP4: 4-bit E2M1 codes with one E4M3 block scale per 16 consecutive
 * weights along K, plus one FP32 scale g per weight tensor. The activation x is bf16.
 * Accumulation is in fp32 and the output is fp32 or bf16. Sources:
 *   - "glm-5.3-flash-nvfp4-tp3-512k--gb10 card.json", performance[4], [6], [8], [9] and
 *     [33], field `note`: the W4A16 GEMV kernels read an NVFP4 weight (E2M1 elements and a
 *     UE4M3 scale per 16) and a BF16 activation;
 *   - "glm-5.3-flash-nvfp4-tp3-512k--gb10 graph.json", node l0.kda.q, `steps`: bf16
 *     activation; the nvfp4/g16 weight is widened to bf16; bf16 x bf16 products are
 *     accumulated in f32; an f32 scale is applied last;
 *   - "GLM-5.3-Flash-NVFP4" blueprint page, section Precision: nvfp4/g16 weight with
 *     bf16 activation is the most common weighted-node format.
 *
 * Layout (a reading: the pages fix none of it):
 *   - w_packed [N, K/2] bytes, row-major. Element 2j of a row is the LOW nibble of byte j.
 *   - w_scales [N, K/16] bytes, row-major, no swizzle. Byte b covers elements 16b..16b+15.
 *   - x [M, K] bf16 (passed as uint16 bit patterns), row-major, rows K elements apart.
 *   - y [M, ldy] with ldy = N (gate_up: 2N; MoE: one row of N per slot), fp32 or bf16.
 *   - Scale codes 0x7F and 0xFF are NaN and propagate to their output column.
 *
 * Ownership and execution:
 *   - Every pointer is caller-owned DEVICE memory on the current CUDA device, except
 *     where a comment says otherwise. The library frees nothing it did not allocate.
 *   - A call allocates no memory and does not synchronise. It validates its arguments on
 *     the host, enqueues its kernel(s) on `stream` (a cudaStream_t; NULL = legacy default
 *     stream) and returns. Calls that take all their memory from the caller can be captured
 *     into CUDA graphs.
 *   - Shapes: 0 <= M <= 8, N >= 0, K >= 0, K % 16 == 0. M == 0, N == 0 or an empty MoE
 *     routing launch nothing. K == 0 sets y to zero.
 *   - Fast path: w/s base pointers 16-byte aligned and K % 32 == 0. Anything else runs a
 *     slower kernel with byte loads, which gives the same results within tolerance.
 *
 * Errors: a non-zero nvfp4_status is returned before anything is enqueued, except
 * NVFP4_ERR_CUDA (a launch error reported by the runtime after the launch). Problems that
 * are only visible on the device (an out-of-range expert id, a pipeline wait that ran
 * past its time budget) never trap. They set bits in a device status word that
 * nvfp4_device_status() reads, and they leave the affected outputs unspecified (bad ids:
 * zero).
 */
#ifndef NVFP4_GEMV_H_
#define NVFP4_GEMV_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    NVFP4_OK = 0,
    NVFP4_ERR_NULL = 1,        /* a required pointer is NULL */
    NVFP4_ERR_SHAPE = 2,       /* M > 8, negative size, K % 16 != 0, top_k/T/E invalid */
    NVFP4_ERR_ALIGN = 3,       /* an FFN workspace not 256-byte aligned (other misalignment runs
                                  the byte-load kernel) */
    NVFP4_ERR_DTYPE = 4,       /* y_type is not one of nvfp4_out_t */
    NVFP4_ERR_UNSUPPORTED = 5, /* a size beyond what any kernel here can take */
    NVFP4_ERR_CUDA = 6,        /* the CUDA runtime reported an error (see nvfp4_last_cuda_error) */
    NVFP4_ERR_TIMEOUT = 7      /* reported by nvfp4_device_status(): a device wait timed out */
} nvfp4_status;

typedef enum {
    NVFP4_OUT_F32 = 0,
    NVFP4_OUT_BF16 = 1         /* round to nearest even from the fp32 result */
} nvfp4_out_t;

/* Device status bits (see nvfp4_device_status). */
#define NVFP4_DEV_TIMEOUT 1    /* a pipeline wait exceeded its time budget; y unspecified */
#define NVFP4_DEV_BAD_EXPERT 2 /* an expert id outside [0, E); those slots are zero */
#define NVFP4_DEV_INTERNAL 4   /* a launch-plan invariant failed on the device; y unspecified */

/*
 * Dense GEMV: y[M, N] = g * W[N, K] . x[M, K]^T (per element as above).
 *   w_packed [N, K/2] u8, w_scales [N, K/16] u8, global_scale = g (by value),
 *   x [M, K] bf16 bits, y [M, N] of y_type.
 * This is the M = 1..8 decode projection GEMV (w4a16_gemv_pipe_m1/_m2 family,
 * "glm-5.3-flash-nvfp4-tp3-512k--gb10 card.json" performance[6], [8]), for example
 * attention projections of the shapes in "llama.cpp eval-callback — ggml op level"
 * (MUL_MAT attn_q {4096, 4096}, attn_k/attn_v {4096, 1024}).
 */
nvfp4_status nvfp4_gemv(const uint8_t* w_packed, const uint8_t* w_scales, float global_scale,
                        const uint16_t* x, void* y, nvfp4_out_t y_type,
                        int M, int N, int K, void* stream);

/*
 * Gate and up projections in one launch (the fused "gate|up N=768+768" projection of
 * "glm-5.3-flash-nvfp4-tp3-512k--gb10 card.json" performance[9]):
 *   y[m, 0:N]  = g_gate * W_gate . x[m],   y[m, N:2N] = g_up * W_up . x[m].
 * Each weight is [N, K/2] + [N, K/16] with its own global scale. y is [M, 2N].
 */
nvfp4_status nvfp4_gemv_gate_up(const uint8_t* w_gate, const uint8_t* s_gate, float g_gate,
                                const uint8_t* w_up, const uint8_t* s_up, float g_up,
                                const uint16_t* x, void* y, nvfp4_out_t y_type,
                                int M, int N, int K, void* stream);

/*
 * Gate and up projections with the activation fused into the epilogue (the swiglu_clamp
 * and silu_mul nodes that follow the gate/up projection in "glm-5.3-flash-nvfp4-tp3-512k--gb10
 * graph.json", block l0.mlp, both "compute f32"; the shared expert's fused group of the same
 * graph). With gate and up as nvfp4_gemv_gate_up computes them (fp32),
 *     c(v)    = min(max(v, -clamp_limit), clamp_limit)   (NaN stays NaN)
 *     y[m, n] = silu(c(gate[m, n])) * c(up[m, n]),   silu(v) = v / (1 + exp(-v)),
 * evaluated in fp32 and stored as y_type. y is [M, N]: the [M, 2N] gate|up product is never
 * written. clamp_limit must be > 0; +INFINITY means no clamp. The pages name the clamp but
 * give no limit, so the limit is the caller's. Returns NVFP4_ERR_SHAPE for clamp_limit <= 0
 * or NaN. Other arguments, errors and layouts as nvfp4_gemv_gate_up.
 */
nvfp4_status nvfp4_gemv_gate_up_swiglu(const uint8_t* w_gate, const uint8_t* s_gate, float g_gate,
                                       const uint8_t* w_up, const uint8_t* s_up, float g_up,
                                       const uint16_t* x, float clamp_limit, void* y, nvfp4_out_t y_type,
                                       int M, int N, int K, void* stream);

/*
 * The FFN block as one call: the shared-expert group of "glm-5.3-flash-nvfp4-tp3-512k--gb10
 * graph.json" (block l3.moe, nodes shared_gate_up, shared_clamp, shared_act and shared_down, which
 * the plan runs as one fused group):
 *     h[m, i] = bf16(silu(c(gate[m, i])) * c(up[m, i]))        (nvfp4_gemv_gate_up_swiglu, bf16)
 *     y[m, n] = g_down * sum_i W_down[n, i] * h[m, i]          (nvfp4_gemv on h)
 * with gate = g_gate * W_gate . x and up = g_up * W_up . x in fp32, and h rounded to nearest
 * even (the silu_mul node's bf16 output).
 *   w_gate, w_up [I, H/2] and s_gate, s_up [I, H/16]; w_down [H, I/2] and s_down [H, I/16];
 *   x [M, H] bf16 bits; y [M, H] of y_type. clamp_limit as nvfp4_gemv_gate_up_swiglu.
 *   workspace: caller-owned device memory of nvfp4_ffn_workspace_bytes(M, I) bytes, 256-byte
 *   aligned (else NVFP4_ERR_ALIGN). Its first 2048 bytes are counters (finished CTAs, and how
 *   much of each slice of h is written): they must be zero before the first call that uses the
 *   workspace, and every call leaves them at zero for the next. h [M, I] bf16 follows at byte
 *   2048. Calls that share a workspace must be ordered (one stream, or events): two in flight at
 *   once corrupt each other's h and counters.
 * Shapes: 0 <= M <= 8, H, I >= 0, H % 16 == 0, I % 16 == 0. M == 0 or H == 0 launch nothing;
 * I == 0 sets y to zero.
 * Execution: one launch when H % 512 == 0, I % 512 == 0, the weights and x are 16-byte aligned,
 * the three weights take at most 12 MiB (3 * H * I * 9/16 bytes; larger blocks are faster as two
 * launches) and a plan with two CTAs per SM fits in shared memory (the shared expert H = 4096,
 * I = 768: M = 1 to 4). That launch runs gate/up and the activation, then down, whose warps each
 * wait only until the slice of h they read is complete (the gate/up items that write it count
 * themselves in the workspace) and whose first weight copies are in flight before that. It needs
 * all its CTAs resident at once; if other work on the GPU keeps some of them from starting
 * within the wait budget, the call sets NVFP4_DEV_TIMEOUT and y is unspecified. Otherwise two
 * launches (gate/up + activation into the workspace's h, then down), with the same results
 * within tolerance.
 */
nvfp4_status nvfp4_ffn_swiglu(const uint8_t* w_gate, const uint8_t* s_gate, float g_gate,
                              const uint8_t* w_up, const uint8_t* s_up, float g_up,
                              const uint8_t* w_down, const uint8_t* s_down, float g_down,
                              const uint16_t* x, float clamp_limit, void* workspace,
                              void* y, nvfp4_out_t y_type, int M, int H, int I, void* stream);

/* Bytes of workspace nvfp4_ffn_swiglu needs: 2048 + M * I * 2 rounded up to 256; -1 when M is
 * outside 0..8 or I < 0. */
int64_t nvfp4_ffn_workspace_bytes(int M, int I);

/*
 * nvfp4_ffn_swiglu without a caller workspace: the same operation and arguments, with the
 * workspace taken from a 256 KB array in the library's own device memory (one per device and
 * process), so the call allocates nothing and needs nothing allocated by the caller. This entry
 * point has no counterpart in the source pages: it is for callers that cannot provide a workspace,
 * such as a C caller with no device allocator of its own, or one whose allocator must not run on
 * its decode path.
 *   Limit: nvfp4_ffn_workspace_bytes(M, I) <= 262144 (M * I <= 130048: M = 8 at I = 12288);
 *   larger returns NVFP4_ERR_UNSUPPORTED before anything is enqueued.
 *   Set-up: the first call on a device looks the array up (cudaGetSymbolAddress) and zeroes its
 *   counters on `stream`; make that first call before any stream capture on the device.
 *   Races: every call on a device uses the same array, so calls must not overlap in time (keep
 *   them on one stream, or order them with events); overlapping calls corrupt each other's h and
 *   counters.
 */
nvfp4_status nvfp4_ffn_swiglu_static(const uint8_t* w_gate, const uint8_t* s_gate, float g_gate,
                                     const uint8_t* w_up, const uint8_t* s_up, float g_up,
                                     const uint8_t* w_down, const uint8_t* s_down, float g_down,
                                     const uint16_t* x, float clamp_limit, void* y, nvfp4_out_t y_type,
                                     int M, int H, int I, void* stream);

/*
 * Routed-expert GEMV over slots (w4a16_gemv_sw_moe, "glm-5.3-flash-nvfp4-tp3-512k--gb10
 * card.json" performance[33]: routed gate or up, 8 slots). For slot s = t*top_k + j
 * (token-major), with e = expert_ids[s]:
 *     y[s, n] = global_scales[e] * sum_k W_e[n, k] * x[r, k],  r = s if x_per_slot else t.
 *   w_packed [E, N, K/2], w_scales [E, N, K/16]: all experts' weights back to back.
 *   global_scales [E] f32 (device), expert_ids [T*top_k] int32 (device).
 *   x [T, K] (x_per_slot = 0: gate/up, shared by a token's slots) or [T*top_k, K]
 *   (x_per_slot = 1: down, one row per slot). y [T*top_k, N].
 * Slots routed to the same expert share reads of that expert's weights: one read serves up to
 * 8 of its slots (the tensor-core tile's 8 columns), so an expert with at most 8 slots in the
 * call is read once (the union of the routed experts, as in glm5next_moe_row_union, card
 * performance[31]), one with more once per 8 of them.
 * An id outside [0, E) zeroes its slot's row and sets NVFP4_DEV_BAD_EXPERT in the device
 * status word and, if status_dev is not NULL, in *status_dev (device int32, OR-ed in).
 */
nvfp4_status nvfp4_moe_gemv(const uint8_t* w_packed, const uint8_t* w_scales,
                            const float* global_scales, int E,
                            const int32_t* expert_ids, int T, int top_k,
                            const uint16_t* x, int x_per_slot,
                            void* y, nvfp4_out_t y_type, int N, int K,
                            int32_t* status_dev, void* stream);

/*
 * Scale-dictionary NVFP4 ("glm-5.3-flash-nvfp4-tp3-512k--gb10 card.json", performance[64],
 * note: routed gate+up weights at 4.3125 bit/weight with a scale dictionary, a tensor kept
 * plain at 4.5). The E2M1 codes are as above; each 16-element block's E4M3 scale code is
 * dict[index] for a 5-bit index and a per-tensor table `scale_dict` of 32 E4M3 codes, so a
 * weight costs 4 + 5/16 bits. The pages give only the bit budget; the layout is this library's
 * reading:
 *   - K % 256 == 0. The index plane has nvfp4_sdict_plane_bytes(N, K) bytes: one 160-byte
 *     record per 16-row tile r (N rounded up to a multiple of 16) and 256-column segment c, at
 *     byte (r * (K / 256) + c) * 160. The index of (row 16r + i, block 16c + j) sits at
 *     position q = 16 i + j as bits 5q .. 5q + 4 of the record, least significant first, where
 *     bit p of a record is bit p % 8 of byte p / 8. Indices of padding rows are ignored.
 *   - A tensor whose block scales take more than 32 distinct codes has no dictionary form (it
 *     stays plain), so the product equals nvfp4_gemv's on the scales dict[index], exactly up
 *     to the fp32 summation order.
 * The index plane must be 16-byte aligned for the tile kernel (else the byte-load kernel
 * runs); the table has no alignment rule. Both are weights: the kernel reads them before the
 * dependency wait (see nvfp4_set_pdl).
 */

/*
 * Dense GEMV with dictionary scales: w_packed [N, K/2], scale_idx (index plane), scale_dict
 * [32] E4M3 codes, all device memory; otherwise as nvfp4_gemv. Returns NVFP4_ERR_SHAPE when
 * K % 256 != 0.
 */
nvfp4_status nvfp4_gemv_sdict(const uint8_t* w_packed, const uint8_t* scale_idx, const uint8_t* scale_dict,
                              float global_scale, const uint16_t* x, void* y, nvfp4_out_t y_type,
                              int M, int N, int K, void* stream);

/*
 * Routed-expert GEMV with dictionary scales: expert e's index plane starts at
 * scale_idx + e * nvfp4_sdict_plane_bytes(N, K) and its table at scale_dict + 32 e; every
 * other argument, layout and status as nvfp4_moe_gemv. Returns NVFP4_ERR_SHAPE when
 * K % 256 != 0. Up to 256 slots run the stream-K tile kernel (each CTA inside one expert group,
 * so one table serves it); larger routings run the byte-load kernel.
 */
nvfp4_status nvfp4_moe_gemv_sdict(const uint8_t* w_packed, const uint8_t* scale_idx, const uint8_t* scale_dict,
                                  const float* global_scales, int E, const int32_t* expert_ids, int T, int top_k,
                                  const uint16_t* x, int x_per_slot, void* y, nvfp4_out_t y_type, int N, int K,
                                  int32_t* status_dev, void* stream);

/* Bytes of the index plane of one [N, K] tensor, or -1 when N < 0, K < 0 or K % 256 != 0. */
int64_t nvfp4_sdict_plane_bytes(int N, int K);

/*
 * Host-side encoder (no GPU): from plain E4M3 block scales [N, K/16] (host memory) writes the
 * index plane (plane_out, nvfp4_sdict_plane_bytes(N, K) bytes of host memory) and the table
 * (dict_out, 32 bytes): the distinct codes in increasing byte order, the rest of the table
 * filled with the last one. Returns the number of distinct codes (0..32), -1 when there are
 * more than 32 (the tensor stays plain; the outputs are not written), or -2 for a bad argument
 * (NULL dict_out, NULL scales or plane_out for a non-empty tensor, negative size, K % 256 != 0).
 */
int nvfp4_sdict_encode(const uint8_t* scales, int N, int K, uint8_t* plane_out, uint8_t* dict_out);

/* Human-readable name of a status code. The returned string is static. */
const char* nvfp4_status_string(int status);

/* The last CUDA runtime error code seen by this library in the calling process (0 = none). */
int nvfp4_last_cuda_error(void);

/*
 * Reads and clears the library's device status word for the current device. It
 * synchronises `stream` first. *flags_out (host memory) receives NVFP4_DEV_* bits.
 * Returns NVFP4_OK, NVFP4_ERR_TIMEOUT if the timeout bit was set, or NVFP4_ERR_CUDA.
 */
nvfp4_status nvfp4_device_status(int32_t* flags_out, void* stream);

/*
 * Time budget of every device-side pipeline wait, in nanoseconds (process-wide; default
 * 1e9). A wait that runs past it makes the kernel set NVFP4_DEV_TIMEOUT, drain the copies
 * it has in flight and return. Passing 0 forces the timeout path (used by tests).
 * Passing UINT64_MAX restores the default.
 */
void nvfp4_set_wait_budget_ns(uint64_t ns);

/*
 * Kernel selection (process-wide): 0 = automatic (default), 1 = always the byte-load
 * kernel, 2 = automatic kernel with the exact fp32 x path forced (the path a CTA takes
 * when x cannot be staged exactly in f16), 3 = the bulk-copy streaming kernel even where
 * the warp-tile kernel applies. Used by tests to check every path against the oracle.
 * The environment variable NVFP4_GEMV_FORCE_VARIANT (0..3) sets the value the library starts
 * with; anything else there is ignored.
 */
void nvfp4_set_variant(int variant);

/*
 * The streaming kernel feeds the tensor cores x in f16, with one power-of-two scale per x
 * row. That is exact for every bf16 value within 2^26 of its row's largest magnitude. A
 * CTA that finds a value it cannot hold exactly (a huge dynamic range inside a row, Inf or
 * NaN) computes with x in fp32 on the CUDA cores instead. This returns how many CTAs did
 * so since the last call, after synchronising `stream`, and resets the count. Returns -1
 * on a CUDA error.
 */
long long nvfp4_fp32_fallbacks(void* stream);

/*
 * Programmatic dependent launch (process-wide; default 1 = on). When on, each GEMV kernel
 * lets the next kernel in the stream start early, and it starts streaming its own weights
 * before the preceding kernel has finished. x, the expert ids and y are touched only after
 * the preceding kernel completes. Weights therefore must not be written by the kernel that
 * immediately precedes the call on the same stream. 0 turns this off: every launch then
 * waits for the full completion of its predecessor.
 */
void nvfp4_set_pdl(int enable);

/*
 * Describes the launch the next call with these arguments would make. It writes
 * "kernel grid block smem split rows_per_item k_warps ..." into buf (host memory,
 * NUL-terminated). kind: 0 dense, 1 gate_up, 2 MoE with x shared by a token's slots,
 * 3 MoE with one x row per slot, 4 gate_up with the fused activation, 5 dense with dictionary
 * scales, 6 and 7 MoE with dictionary scales (x shared / one x row per slot), 8 the FFN block
 * (nvfp4_ffn_swiglu with N = H, K = I); for the MoE kinds M is the number of experts E.
 * Pointers are assumed 256-byte aligned. Returns the number of characters, or -1.
 */
int nvfp4_describe_plan(int kind, int M, int N, int K, int T, int top_k, char* buf, int buflen);

/*
 * nvfp4_describe_plan for a described device instead of the current one: sm_count SMs,
 * smem_optin bytes of shared memory a CTA may opt into, smem_per_sm bytes per SM. It runs the
 * planner on the host only (no GPU or driver needed) and assumes the tile kernel's TMA
 * tensor-map encoder is available. Returns the number of characters, or -1 for a bad
 * argument (kind outside 0..8, sizes < 1, smem_per_sm < smem_optin).
 */
int nvfp4_describe_plan_host(int sm_count, int smem_optin, int smem_per_sm, int kind, int M, int N, int K,
                             int T, int top_k, char* buf, int buflen);

/*
 * Phase trace of the tile kernels (a diagnostic; no counterpart on the pages). A library built
 * with -DNVFP4_PHASE_TRACE=1 records, for each of the last 16 tile-kernel launches (slot =
 * launch number mod 16) and each of its first 1024 CTAs, 40 64-bit words: for phase ph = 0..7
 * word 2ph is %globaltimer (ns) and word 2ph + 1 the SM's clock64, taken by thread 0 at
 * 0 entry, 1 first weight copies issued, 2 past the dependency wait, 3 x staged, 4 first box
 * landed, 5 box loop done (stream-K form), 6 outputs stored, 7 exit; word 16 + w is
 * %globaltimer when warp w left its box loop; word 24 the SM id; word 24 + w (w = 1..7)
 * %globaltimer when warp w's first box landed; words 32..37 thread 0's clock64 when the barriers
 * were initialised, the work range known, the first and all initial weight copies issued
 * (dense launches), the MoE groups built, and the copies that follow x staging issued. Words 38
 * and 39: dense launches, thread 0's clock64 just before and just after its first box wait; MoE
 * launches, the group builder's steps; the FFN block, its slice of h complete and staged. A
 * build with -DNVFP4_TRACE_BOX_LANDED=1 also has thread 0 of a dense launch wait for its first
 * box before the dependency wait and record %globaltimer then in word 36. Phase 3 is taken right
 * after x staging. Unrecorded words are zero.
 * This call synchronises `stream`, copies min(max_words, 16 * 1024 * 40) words in
 * [slot][cta][word] order to host_out (host memory), clears the trace and restarts the slot
 * count. Returns the number of words copied, 0 for a library built without tracing (the
 * default), or -1 on a CUDA error or a NULL host_out.
 */
int nvfp4_phase_trace(uint64_t* host_out, int max_words, void* stream);

/* Library version: major * 10000 + minor * 100 + patch. */
int nvfp4_version(void);

#ifdef __cplusplus
}
#endif

#endif /* NVFP4_GEMV_H_ */
