// NVFP4 (nvfp4/g16) weight-only GEMV for GB300 (sm_103a): kernels and the C ABI.
//
//   y[m, n] = g * sum_k E2M1(q[n, k]) * E4M3(s[n, k / 16]) * x[m, k]      (m < M <= 8)
//
// This is the decode-time W4A16 projection GEMV ("glm-5.3-flash-nvfp4-tp3-512k--gb10
// card.json", performance[6], [8], [9], [33]: W4A16 NVFP4 weight with E2M1 elements and
// a UE4M3 scale per 16, BF16 activation). Each term follows node l0.kda.q of
// "glm-5.3-flash-nvfp4-tp3-512k--gb10 graph.json": the weight is widened, multiplied by
// the bf16 activation and accumulated in f32, and the f32 tensor scale is applied last.
//
// Kernels:
//   * gemv_tile_kernel (default for K % 256 == 0, aligned operands; dense, gate/up and up to
//     32 MoE slots): every warp owns 16-row tiles and keeps its own ring of TMA tensor copies
//     (128-byte swizzled codes + scales) full; the products run on the tensor cores as
//     mma.sync.m16n8k16 with the weights decoded exactly to f16 (E2M1 * E4M3) and x staged in
//     f16 per K slice. K may be split over warps (shared-memory reduction) or over a cluster
//     (DSMEM reduction), both in a fixed order. See the comment above the kernel. Its third
//     template flag gives gate/up with the fused SwiGLU: gate and up tiles alternate, so a
//     pair meets in shared memory and only silu(clamp(gate)) * clamp(up) is stored.
//   * gemv_tile_sk_kernel (MoE launches with many tiles per CTA): the same warp rings and
//     decode in a stream-K form. Whole (expert group, tile) jobs are spread evenly over the
//     CTAs and their TMA boxes evenly over each CTA's warps; a job cut between warps is
//     summed in a fixed warp order.
//   * gemv_stream_kernel (K % 32 == 0 otherwise, or up to 256 MoE slots): a producer warp
//     bulk-copies whole items of rows into a ring, consumer warps decode with the same MMA
//     scheme and an epilogue warp reduces in a fixed order.
//   * gemv_simple_kernel: byte loads for every other alignment and size.
// Every mbarrier wait is bounded by a %globaltimer budget. On expiry a kernel sets a device
// status bit, drains the copies it has in flight and finishes: it never traps.

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>

#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <type_traits>
#include <mutex>

#include "nvfp4_gemv.h"

namespace nvfp4 {

constexpr int kConsumerWarps = 8;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kEpilogueWarp = kConsumerWarps + 1;
constexpr int kThreads = (kConsumerWarps + 2) * 32;
constexpr int kMaxStages = 4;
constexpr int kStageData = 60 * 1024;      // most weight bytes (codes + scales) per stage
constexpr int kStepElems = 1024;           // K elements per warp step (32 lanes x 32)
constexpr int kMaxMoeSlots = 256;
constexpr int kSimpleThreads = 256;
constexpr uint64_t kDefaultWaitNs = 1000000000ull;
constexpr uint64_t kDrainWaitNs = 2000000000ull;

enum : int { kModeDense = 0, kModeMoe = 1 };

__device__ int g_device_status;
__device__ unsigned long long g_fp32_fallbacks;  // CTAs that staged x in fp32 because f16 was inexact

// Phase trace (diagnostic builds with -DNVFP4_PHASE_TRACE=1 only): the tile kernels write, per
// launch slot and CTA, kTraceWords 64-bit words: for phase ph = 0..7 word 2ph = %globaltimer (ns)
// and word 2ph + 1 = clock64 (thread 0); word 16 + w = %globaltimer when warp w leaves its box
// loop; word 24 = the SM the CTA ran on; word 24 + w (w = 1..7) = %globaltimer when warp w's
// first box landed (warp 0's is phase 4); words 32.. = clock64 of thread 0 at finer points of
// the prologue (32 barriers initialised, 33 work range known, 34 first copy issued, 35 all
// initial copies issued, 36 MoE groups built, 37 copies after x staging issued; the FFN block:
// 38 its slice of h complete, 39 that slice staged; MoE with more than 32 slots: 38 ids in
// shared memory, 39 ranks and counts done; with up to 32: 38 warp 0's groups built, 39 the CTA
// past the barrier after them; dense tile launches: 38 just before and 39 just after warp 0's
// wait for its first box, and with -DNVFP4_TRACE_BOX_LANDED=1 word 36 = %globaltimer when that
// box, requested before the dependency wait, landed). Phases: 0 entry, 1 first weight copies issued, 2 past
// the dependency wait, 3 x staged, 4 warp 0's first box landed, 5 warp 0's loop done, 6 outputs
// stored, 7 exit. Normal builds compile all of it out.
#ifndef NVFP4_PHASE_TRACE
#define NVFP4_PHASE_TRACE 0
#endif
#ifndef NVFP4_TRACE_BOX_LANDED
#define NVFP4_TRACE_BOX_LANDED 0  // traced builds: dense word 36 = %globaltimer when the first box landed
#endif
constexpr int kTraceLaunches = 16;
constexpr int kTraceCtas = 1024;
constexpr int kTraceWords = 40;
#if NVFP4_PHASE_TRACE
__device__ unsigned long long g_trace[kTraceLaunches * kTraceCtas * kTraceWords];
// The CTA's words collect in shared memory and go to g_trace at exit (trace_flush): a global
// store here would hold up the next release-ordered operation (an mbarrier fence or arrive) for
// its round trip and so distort the phases it measures.
__shared__ unsigned long long s_trace[kTraceWords];
#endif

// ------------------------------------------------------------------ parameters

struct Params {
    const uint8_t* w[2];      // dense: weight codes per group (gate, up); MoE: w[0] = all experts
    const uint8_t* s[2];      // scales, same layout
    float g[2];               // dense global scales
    const float* g_dev;       // MoE per-expert global scales
    const int32_t* ids;       // MoE expert ids [slots]
    int32_t* status_user;     // MoE optional status word
    const uint16_t* x;        // bf16 bits
    void* y;
    int64_t ldy;              // output row stride in elements
    int out_bf16;
    int M, N, K;
    int groups;               // dense: 1 or 2
    int E, T, top_k, x_per_slot, slots;
    int S, Kr, J;             // K split (cluster size), K per CTA, warp steps per CTA K-range
    int rpi, chunks, items;   // rows per item, items per group, items in total (dense)
    int items_q, items_r;     // dense: items / units and items % units (units = CTAs or clusters)
    int s_aligned;            // scale rows are whole 16-byte lines (K % 256 == 0, aligned bases)
    int ck, cr;               // consumer warps along K and along rows
    int mstride;              // partial-sum stride per row (>= max rows of x per item)
    int cl_rows;              // rows of the cluster partial buffer (S > 1)
    int stages;               // ring depth (2..kMaxStages)
    uint32_t stage_stride;    // bytes per ring slot (multiple of 128)
    long long work;           // planner's estimate of decoded row-elements per unit (host only)
    int force_f32;            // 1: always stage x in fp32 (kernel selection for tests)
    int wstride;              // bytes between weight rows in a ring slot (padded: 64 mod 128)
    int xh_stride;            // bytes between staged f16 x rows (tensor-core path; 64 mod 128)
    uint32_t x_off, xraw_off, misc_off, red_off, cl_off, bar_off, tab_off;
    uint64_t wait_ns;
};

struct MoeTables {
    int n_groups;
    int pad_[3];
    int expert[kMaxMoeSlots];
    int count[kMaxMoeSlots];
    int first[kMaxMoeSlots];                  // index into member_list
    int member_list[kMaxMoeSlots];            // slots grouped by expert, slot order
};

// ------------------------------------------------------------------ PTX helpers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
    asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;"
                 ::"r"(smem_addr(bar)), "r"(bytes) : "memory");
}

// The suspend-time hint lets a waiting warp sleep until the phase completes (or the hint
// elapses) instead of spinning on issue slots that the decoding warps need.
constexpr uint32_t kSuspendHintNs = 1000000;

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2, %3;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity), "n"(kSuspendHintNs) : "memory");
    return ok != 0;
}

__device__ __forceinline__ bool mbar_test_wait(uint64_t* bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n"
        " mbarrier.test_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok) : "r"(smem_addr(bar)), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait for the phase with the given parity; false when the budget ran out.
// A zero budget polls once without blocking (try_wait may suspend for a while).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, uint64_t budget_ns) {
    if (budget_ns == 0) return mbar_test_wait(bar, parity);
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    while (true) {
        if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > budget_ns) return false;
    }
}

// TMA bulk copy global -> shared (this CTA), completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_g2s(void* dst, const void* src, uint32_t bytes, uint64_t* bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
        ::"r"(smem_addr(dst)), "l"(src), "r"(bytes), "r"(smem_addr(bar)) : "memory");
}

__device__ __forceinline__ uint4 lds128(uint32_t a) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(a));
    return v;
}

__device__ __forceinline__ float4 lds128f(uint32_t a) {
    float4 v;
    asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(a));
    return v;
}

__device__ __forceinline__ uint16_t lds16(uint32_t a) {
    uint16_t v;
    asm volatile("ld.shared.u16 %0, [%1];" : "=h"(v) : "r"(a));
    return v;
}

__device__ __forceinline__ float2 lds64f(uint32_t a) {
    float2 v;
    asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(a));
    return v;
}

// Programmatic dependent launch: wait for the preceding kernel's results / let the next
// kernel start its prologue. Both are no-ops when the launch did not enable PDL.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n"
                 "barrier.cluster.wait.acquire.aligned;" ::: "memory");
}

__device__ __forceinline__ float ld_cluster_f32(const float* local, uint32_t rank) {
    uint32_t remote;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(remote) : "r"(smem_addr(local)), "r"(rank));
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(remote) : "memory");
    return v;
}

// Four E2M1 pairs (one 32-bit word, 8 codes; element 2i in the low nibble of byte i) ->
// four f16x2 (low half = even element). Exact: every E2M1 value is an f16.
__device__ __forceinline__ void cvt_e2m1x8(uint32_t w, uint32_t (&h)[4]) {
    asm("{\n .reg .b8 b0, b1, b2, b3;\n"
        " mov.b32 {b0, b1, b2, b3}, %4;\n"
        " cvt.rn.f16x2.e2m1x2 %0, b0;\n"
        " cvt.rn.f16x2.e2m1x2 %1, b1;\n"
        " cvt.rn.f16x2.e2m1x2 %2, b2;\n"
        " cvt.rn.f16x2.e2m1x2 %3, b3;\n}"
        : "=r"(h[0]), "=r"(h[1]), "=r"(h[2]), "=r"(h[3]) : "r"(w));
}

// Two E4M3 scale codes (low byte = first block) -> f16x2. Exact: E4M3 values are f16s.
__device__ __forceinline__ uint32_t cvt_e4m3x2(uint16_t v) {
    uint32_t d;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"(v));
    return d;
}

// (lo(h2) * s, hi(h2) * s) in fp32. E2M1 * E4M3 has at most 6 significant bits, so the
// products are exact: this is the weight widened to full precision.
__device__ __forceinline__ float2 widen_scaled(uint32_t h2, uint16_t s) {
    float2 r;
    asm("{\n .reg .f16 a, b;\n"
        " mov.b32 {a, b}, %2;\n"
        " fma.rn.f32.f16 %0, a, %3, 0f00000000;\n"
        " fma.rn.f32.f16 %1, b, %3, 0f00000000;\n}"
        : "=f"(r.x), "=f"(r.y) : "r"(h2), "h"(s));
    return r;
}

// acc + lo(q2) * lo(x2) + hi(q2) * hi(x2): two mixed-precision FMAs (f16 x f16 products,
// exact in fp32, accumulated in fp32).
__device__ __forceinline__ float fma2_f16_f32(uint32_t q2, uint32_t x2, float acc) {
    float r;
    asm("{\n .reg .f16 a, b, c, d;\n"
        " mov.b32 {a, b}, %1;\n"
        " mov.b32 {c, d}, %2;\n"
        " fma.rn.f32.f16 %0, a, c, %3;\n"
        " fma.rn.f32.f16 %0, b, d, %0;\n}"
        : "=f"(r) : "r"(q2), "r"(x2), "f"(acc));
    return r;
}

__device__ __forceinline__ float half_lo_f32(uint32_t h2) { return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 & 0xffffu))); }
__device__ __forceinline__ float half_hi_f32(uint32_t h2) { return __half2float(__ushort_as_half(static_cast<unsigned short>(h2 >> 16))); }

// f16x2 product. E2M1 * E4M3 has at most 6 significant bits and stays in the f16 normal
// range, so this is the exact dequantised weight pair.
__device__ __forceinline__ uint32_t hmul2_u32(uint32_t a, uint32_t b) {
    uint32_t d;
    asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t sel) {
    uint32_t d;
    asm("prmt.b32 %0, %1, 0, %2;" : "=r"(d) : "r"(a), "r"(sel));
    return d;
}

// ------------------------------------------------------------------ scale dictionary
// Scale-dictionary NVFP4 ("glm-5.3-flash-nvfp4-tp3-512k--gb10 card.json", performance[64],
// note: routed experts at 4.3125 bit/weight with a scale dictionary): each 16-element block's
// E4M3 scale code is dict[index] for a 5-bit index and a 32-entry table per tensor. Index plane
// layout (K % 256 == 0): one 160-byte record per 16-row tile r and 256-column segment c at byte
// (r * K/256 + c) * 160; (row 16r + i, block 16c + j) at q = 16i + j, bits 5q .. 5q + 4, least
// significant first, bit p of a record being bit p % 8 of byte p / 8.
constexpr int kSdRecord = 160;     // bytes of one (tile, segment) record
constexpr int kSdPairs = 1024;     // entries of the pair table: two 5-bit indices

__host__ __device__ __forceinline__ int64_t sd_plane_bytes(int64_t N, int64_t K) {
    return (N + 15) / 16 * (K / 256) * kSdRecord;
}

// The scale code of block b of row n (byte loads; the byte-load kernel).
__device__ __forceinline__ uint32_t sd_code(const uint8_t* plane, const uint8_t* dict, int64_t K, int64_t n,
                                            int64_t b) {
    const uint8_t* rec = plane + ((n >> 4) * (K >> 8) + (b >> 4)) * kSdRecord;
    const uint32_t bit = static_cast<uint32_t>(((n & 15) * 16 + (b & 15)) * 5);
    uint32_t v = __ldg(rec + (bit >> 3));
    if ((bit & 7) > 3) v |= static_cast<uint32_t>(__ldg(rec + (bit >> 3) + 1)) << 8;  // the field spans two bytes
    return __ldg(dict + ((v >> (bit & 7)) & 31u));
}

// D += A * B for one m16n8k16 tile: A 16x16 f16 (row), B 16x8 f16 (col), D 16x8 f32.
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1) {
    asm(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, "
        "{%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ void store_out(void* y, int64_t idx, float v, int out_bf16) {
    if (out_bf16) {
        reinterpret_cast<__nv_bfloat16*>(y)[idx] = __float2bfloat16_rn(v);
    } else {
        reinterpret_cast<float*>(y)[idx] = v;
    }
}

// The fused gate/up activation: silu(clamp(gate)) * clamp(up), both clamped to [-lim, lim]
// (lim = +inf: no clamp), in f32. NaN passes through the clamp. The swiglu_clamp and
// silu_mul nodes of "glm-5.3-flash-nvfp4-tp3-512k--gb10 graph.json" (l0.mlp), whose steps
// read "compute f32".
__device__ __forceinline__ float swiglu_f32(float gate, float up, float lim) {
    gate = gate > lim ? lim : (gate < -lim ? -lim : gate);
    up = up > lim ? lim : (up < -lim ? -lim : up);
    return gate / (1.f + expf(-gate)) * up;
}

__device__ __forceinline__ void trace_word(int slot, int word, unsigned long long v) {
#if NVFP4_PHASE_TRACE
    (void)slot;
    s_trace[word] = v;
#else
    (void)slot; (void)word; (void)v;
#endif
}

// Clears the CTA's trace words (all threads, before any trace_word; ends with __syncthreads).
__device__ __forceinline__ void trace_begin(int tid) {
#if NVFP4_PHASE_TRACE
    if (tid < kTraceWords) s_trace[tid] = 0;
    __syncthreads();
#else
    (void)tid;
#endif
}

// Writes the CTA's trace words to its slot (all threads, at exit).
__device__ __forceinline__ void trace_flush(int slot, int tid) {
#if NVFP4_PHASE_TRACE
    __syncthreads();
    if (tid < kTraceWords && blockIdx.x < kTraceCtas)
        g_trace[(static_cast<size_t>(slot) * kTraceCtas + blockIdx.x) * kTraceWords + tid] = s_trace[tid];
#else
    (void)slot; (void)tid;
#endif
}

// Phase ph of this CTA (call from one thread): %globaltimer and clock64.
__device__ __forceinline__ void trace_phase(int slot, int ph) {
#if NVFP4_PHASE_TRACE
    trace_word(slot, 2 * ph, global_ns());
    trace_word(slot, 2 * ph + 1, static_cast<unsigned long long>(clock64()));
    if (ph == 0) {
        uint32_t sm;
        asm volatile("mov.u32 %0, %%smid;" : "=r"(sm));
        trace_word(slot, 24, sm);
    }
#else
    (void)slot; (void)ph;
#endif
}

__device__ __forceinline__ void raise_status(int bits, int32_t* user) {
    atomicOr(&g_device_status, bits);
    if (user) atomicOr(reinterpret_cast<int*>(user), bits);
}

// ------------------------------------------------------------------ warp reduction

// Transposed butterfly: each lane starts with CNT partials; after the call the sums over
// the 32 lanes are spread across lanes (see lane_owned_*). CNT must be a power of two.
template <int CNT, int O>
__device__ __forceinline__ void reduce_scatter(float* v, int lane) {
    if constexpr (O > 0) {
        if constexpr (CNT > 1) {
            constexpr int H = CNT / 2;
            const bool up = (lane & O) != 0;
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const float send = up ? v[i] : v[i + H];
                const float keep = up ? v[i + H] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, O);
            }
            reduce_scatter<H, O / 2>(v, lane);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], O);
            reduce_scatter<1, O / 2>(v, lane);
        }
    }
}

__host__ __device__ constexpr int next_pow2(int v) { return v <= 1 ? 1 : 2 * next_pow2((v + 1) / 2); }
__host__ __device__ constexpr int ilog2(int v) { return v <= 1 ? 0 : 1 + ilog2(v / 2); }

// ------------------------------------------------------------------ x staging

__device__ __forceinline__ float pow2f(int e) {  // exact 2^e for e in [-149, 127]
    return e >= -126 ? __int_as_float((e + 127) << 23) : __int_as_float(1 << (e + 149));
}

// Byte offset of element k inside a staged f16 x row for the tensor-core path. A row is a
// sequence of 128-element chunks of 256 bytes; within a chunk, the 8 elements
// 32t + 8q .. 32t + 8q + 7 (t, q in 0..3) sit at byte (q * 4 + t) * 16. Lane t of an MMA
// quad then reads its 32 elements with four conflict-free 128-bit loads.
__host__ __device__ __forceinline__ int mma_x_off(int k) {
    return (k >> 7) * 256 + ((((k >> 3) & 3) * 4 + ((k >> 5) & 3)) << 4) + ((k & 7) << 1);
}

__device__ __forceinline__ uint32_t bf16_mag_max(uint4 v) {
    uint32_t a = max(v.x & 0x7fffu, (v.x >> 16) & 0x7fffu);
    a = max(a, max(v.y & 0x7fffu, (v.y >> 16) & 0x7fffu));
    a = max(a, max(v.z & 0x7fffu, (v.z >> 16) & 0x7fffu));
    return max(a, max(v.w & 0x7fffu, (v.w >> 16) & 0x7fffu));
}

// Row-scaled f16 staging for the tensor-core path. The raw bf16 rows of x (this CTA's K
// range) sit in shared memory at xraw, Kr * 2 bytes apart (the producer's bulk copies).
// For each row m one power of two 2^E_m is chosen so that the row's largest |x| lands in
// [2^12, 2^13); x' = x * 2^-E_m is stored as f16 at mma_x_off, rows xstride bytes apart,
// zero-padded to whole 128-element chunks, and e2[m] = 2^E_m. A bf16 value converts
// exactly when x' is zero or a normal f16, i.e. when |x| >= 2^(E_m - 14), at most 2^26
// below the row's largest magnitude. Pass 1 finds each row's largest and smallest nonzero
// magnitude, so the function can return (the same value in every thread) whether any row
// holds a value that would not convert exactly, or Inf/NaN; the caller then uses the fp32
// path. The passes are separated by the consumers' `bar` (bounded wait on `parity`);
// `wmax` is [kConsumerWarps][16] words of scratch. `ok` turns false if that wait times out.
template <int MAXR>
__device__ bool stage_x_mma(const uint8_t* xraw, int Kr, int rows, uint8_t* xh, int xstride, float* e2,
                            uint32_t* wmax, uint64_t* bar, uint32_t parity, uint64_t budget, int tid, int nthreads,
                            bool& ok) {
    const int per_row = Kr / 8;                 // 8-element chunks per row
    const int padded = ((Kr + 127) >> 7) * 16;  // chunks per row including the zero tail
    const int lane = tid & 31, warp = tid >> 5;
    const uint32_t raw = smem_addr(xraw);
    // pass 1: per row, the largest and the smallest nonzero bf16 magnitude (bit patterns of
    // non-negative values order like the values; two per word, compared as 16-bit lanes)
#pragma unroll
    for (int m = 0; m < MAXR; ++m) {
        if (m >= rows) break;
        uint32_t mx = 0u, mn = 0x7fff7fffu;
        for (int c = tid; c < per_row; c += nthreads) {
            const uint4 v = lds128(raw + (m * per_row + c) * 16);
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t mag = w4[i] & 0x7fff7fffu;
                mx = __vmaxu2(mx, mag);
                mn = __vminu2(mn, mag | (__vcmpeq2(mag, 0u) & 0x7fff7fffu));
            }
        }
        uint32_t a = max(mx & 0xffffu, mx >> 16), z = min(mn & 0xffffu, mn >> 16);
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
            z = min(z, __shfl_xor_sync(0xffffffffu, z, o));
        }
        if (lane == 0) {
            wmax[warp * 16 + m] = a;
            wmax[warp * 16 + 8 + m] = z;
        }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar);
    if (!mbar_wait(bar, parity, budget)) {
        ok = false;
        return false;
    }
    bool lossy = false;
#pragma unroll
    for (int m = 0; m < MAXR; ++m) {
        if (m >= rows) break;
        uint32_t amax = 0, amin = 0x7fffu;
        for (int w = 0; w < nthreads / 32; ++w) {
            amax = max(amax, wmax[w * 16 + m]);
            amin = min(amin, wmax[w * 16 + 8 + m]);
        }
        int e_max;
        if (amax >= 0x7f80u || amax == 0) {
            e_max = 12;                        // Inf/NaN (reported below) or an all-zero row
            lossy |= amax >= 0x7f80u;
        } else if ((amax >> 7) == 0) {
            e_max = (31 - __clz(amax)) - 133;  // bf16 subnormal: mant * 2^-133
        } else {
            e_max = static_cast<int>(amax >> 7) - 127;
        }
        const int E = e_max - 12;
        // smallest exact magnitude 2^(E - 14) as a bf16 pattern; bf16 subnormals count as inexact
        const int tb = E - 14 + 127;
        const uint32_t thresh = tb >= 1 ? static_cast<uint32_t>(tb) << 7 : 0x80u;
        lossy |= amin != 0x7fffu && amin < thresh;
        if (tid == 0) e2[m] = pow2f(E);
        // pass 2: x' = x * 2^-E, two f32 -> f16x2 conversions per word
        const int a2 = min(-E, 127);
        const float sa = pow2f(a2), sb = pow2f(-E - a2);  // sb == 1 unless the row is tiny
        for (int c = tid; c < per_row; c += nthreads) {
            const uint4 v = lds128(raw + (m * per_row + c) * 16);
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
            uint32_t out[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __half2 h = __floats2half2_rn(bf16_lo(w4[i]) * sa * sb, bf16_hi(w4[i]) * sa * sb);
                out[i] = *reinterpret_cast<const uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(xh + m * xstride + mma_x_off(c * 8)) = make_uint4(out[0], out[1], out[2], out[3]);
        }
        // zero tail up to the next 128-element chunk
        for (int c = per_row + tid; c < padded; c += nthreads)
            *reinterpret_cast<uint4*>(xh + m * xstride + mma_x_off(c * 8)) = make_uint4(0u, 0u, 0u, 0u);
    }
    return lossy;
}

// ------------------------------------------------------------------ consumer compute

// Reduces V = R * MTE per-lane partials over the warp and stores the sums of rows
// rb..rb+R-1 (those below `rows`) at red[row * mstride + m].
template <int R, int MTE>
__device__ __forceinline__ void store_partials(float (&v)[next_pow2(R * MTE)], int lane, int rb, int rows,
                                               float* red, int mstride) {
    constexpr int V = R * MTE;
    constexpr int VP = next_pow2(V);
    reduce_scatter<VP, 16>(v, lane);
    if constexpr (VP >= 32) {
#pragma unroll
        for (int i = 0; i < VP / 32; ++i) {
            const int idx = lane * (VP / 32) + i;
            if (idx < V) {
                const int row = rb + idx / MTE;
                if (row < rows) red[row * mstride + idx % MTE] = v[i];
            }
        }
    } else {
        constexpr int sh = 5 - ilog2(VP);
        if ((lane & ((1 << sh) - 1)) == 0) {
            const int idx = lane >> sh;
            if (idx < V) {
                const int row = rb + idx / MTE;
                if (row < rows) red[row * mstride + idx % MTE] = v[0];
            }
        }
    }
}

// Exact fp32 path (used when x does not fit the row-scaled f16 staging exactly): one item's
// share of one consumer warp, rows rb = wr*R, wr*R + cr*R, ... in batches of R and
// 1024-element steps j = wk, wk + ck, ... x is read straight from global memory (bf16, L2
// resident); xrow[m] points at row m's element k0. Partials go to
// red[(wk * rpi + row) * mstride + m].
template <int MTE, int R>
__device__ __noinline__ void compute_item_f32(uint32_t wst, uint32_t sst, int wstride, int srow_bytes,
                                                 const uint16_t* const (&xrow)[8], int rows, int Kr, int J, int wr,
                                                 int wk, int cr, int ck, int lane, float* red, int rpi,
                                                 int mstride) {
    constexpr int V = R * MTE;
    constexpr int VP = next_pow2(V);
    for (int rb = wr * R; rb < rows; rb += cr * R) {
        float2 acc[R][MTE];
#pragma unroll
        for (int r = 0; r < R; ++r)
#pragma unroll
            for (int m = 0; m < MTE; ++m) acc[r][m] = make_float2(0.f, 0.f);

        for (int j = wk; j < J; j += ck) {
            const int kl = j * kStepElems + lane * 32;
            if (kl < Kr) {
                uint4 wv[R];
                uint32_t sh[R];
#pragma unroll
                for (int r = 0; r < R; ++r) {
                    const int row = rb + r;
                    if (row < rows) {
                        wv[r] = lds128(wst + row * wstride + (kl >> 1));
                        sh[r] = cvt_e4m3x2(lds16(sst + row * srow_bytes + (kl >> 4)));
                    } else {
                        wv[r] = make_uint4(0u, 0u, 0u, 0u);
                        sh[r] = 0u;
                    }
                }
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    float2 xp[MTE][4];
#pragma unroll
                    for (int m = 0; m < MTE; ++m) {
                        const uint16_t* src = xrow[m] + kl + w * 8;
                        uint32_t u[4];
#pragma unroll
                        for (int i = 0; i < 4; ++i) u[i] = src[2 * i] | (static_cast<uint32_t>(src[2 * i + 1]) << 16);
#pragma unroll
                        for (int i = 0; i < 4; ++i) xp[m][i] = make_float2(bf16_lo(u[i]), bf16_hi(u[i]));
                    }
#pragma unroll
                    for (int r = 0; r < R; ++r) {
                        const uint32_t word = w == 0 ? wv[r].x : (w == 1 ? wv[r].y : (w == 2 ? wv[r].z : wv[r].w));
                        const uint16_t sc = static_cast<uint16_t>(w < 2 ? (sh[r] & 0xffffu) : (sh[r] >> 16));
                        uint32_t h[4];
                        cvt_e2m1x8(word, h);
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            const float2 q = widen_scaled(h[i], sc);
#pragma unroll
                            for (int m = 0; m < MTE; ++m) acc[r][m] = __ffma2_rn(q, xp[m][i], acc[r][m]);
                        }
                    }
                }
            }
        }

        float v[VP];
#pragma unroll
        for (int i = 0; i < VP; ++i) v[i] = i < V ? acc[i / MTE][i % MTE].x + acc[i / MTE][i % MTE].y : 0.f;
        store_partials<R, MTE>(v, lane, rb, rows, red + wk * rpi * mstride, mstride);
    }
}

// One item's share of one consumer warp on the tensor-core path. The item's rows form
// 16-row tiles (the MMA's M); warp (wr, wk) takes tiles wr, wr + cr, ... and 128-element
// K steps wk, wk + ck, ... Lane (g, t) of the MMA quad layout decodes the 32 nibbles
// 32t .. 32t + 31 of each step for rows g and g + 8 (one 128-bit load each). The MMA's
// logical k index is a fixed permutation of these physical positions, and the staged x
// (stage_x_mma) uses the same one, so the dot product is unchanged. A holds
// E2M1 * E4M3 in f16 (exact), B the row-scaled f16 x, D accumulates in f32. The partial
// sums, times each x row's 2^E_m, go to red[(wk * rpi + row) * mstride + m].
template <int MTE>
__device__ __forceinline__ void compute_item_mma(uint32_t wst, int wstride, uint32_t sst, int srow_bytes,
                                                 uint32_t xa, int xstride, const float* e2, int rows, int Kr,
                                                 int wr, int wk, int cr, int ck, int lane, float* red, int rpi,
                                                 int mstride) {
    const int g = lane >> 2, t = lane & 3;
    const int nsteps = (Kr + 127) >> 7;
    const int ntiles = (rows + 15) >> 4;
    const bool xcol = g < MTE;
    const int m0 = 2 * t;
    const float e2a = m0 < MTE ? e2[m0] : 0.f;
    const float e2b = m0 + 1 < MTE ? e2[m0 + 1] : 0.f;
    for (int tile = wr; tile < ntiles; tile += cr) {
        const int ra = tile * 16 + g, rb = ra + 8;
        const bool va = ra < rows, vb = rb < rows;
        const bool upper = tile * 16 + 8 < rows;  // warp-uniform: the tile's rows 8..15 exist
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        for (int j = wk; j < nsteps; j += ck) {
            const int kt = (j << 7) + (t << 5);
            const bool vk = kt < Kr;
            uint4 wa = make_uint4(0u, 0u, 0u, 0u), wb = wa;
            uint32_t sa = 0u, sb = 0u;
            if (vk && va) {
                wa = lds128(wst + ra * wstride + (kt >> 1));
                sa = cvt_e4m3x2(lds16(sst + ra * srow_bytes + (kt >> 4)));
            }
            if (vk && vb) {
                wb = lds128(wst + rb * wstride + (kt >> 1));
                sb = cvt_e4m3x2(lds16(sst + rb * srow_bytes + (kt >> 4)));
            }
            uint4 xq[4];
#pragma unroll
            for (int q = 0; q < 4; ++q)
                xq[q] = xcol ? lds128(xa + g * xstride + (j << 8) + ((q * 4 + t) << 4)) : make_uint4(0u, 0u, 0u, 0u);
            const uint32_t sa0 = prmt(sa, 0x1010u), sa1 = prmt(sa, 0x3232u);
            const uint32_t sb0 = prmt(sb, 0x1010u), sb1 = prmt(sb, 0x3232u);
            if (upper) {
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t ha[4], hb[4];
                    cvt_e2m1x8(w == 0 ? wa.x : (w == 1 ? wa.y : (w == 2 ? wa.z : wa.w)), ha);
                    cvt_e2m1x8(w == 0 ? wb.x : (w == 1 ? wb.y : (w == 2 ? wb.z : wb.w)), hb);
                    const uint32_t s_a = w < 2 ? sa0 : sa1, s_b = w < 2 ? sb0 : sb1;
                    mma_16816(d, hmul2_u32(ha[0], s_a), hmul2_u32(hb[0], s_b), hmul2_u32(ha[1], s_a),
                              hmul2_u32(hb[1], s_b), xq[w].x, xq[w].y);
                    mma_16816(d, hmul2_u32(ha[2], s_a), hmul2_u32(hb[2], s_b), hmul2_u32(ha[3], s_a),
                              hmul2_u32(hb[3], s_b), xq[w].z, xq[w].w);
                }
            } else {  // rows 8..15 of the tile are empty: their A halves are zero
#pragma unroll
                for (int w = 0; w < 4; ++w) {
                    uint32_t ha[4];
                    cvt_e2m1x8(w == 0 ? wa.x : (w == 1 ? wa.y : (w == 2 ? wa.z : wa.w)), ha);
                    const uint32_t s_a = w < 2 ? sa0 : sa1;
                    mma_16816(d, hmul2_u32(ha[0], s_a), 0u, hmul2_u32(ha[1], s_a), 0u, xq[w].x, xq[w].y);
                    mma_16816(d, hmul2_u32(ha[2], s_a), 0u, hmul2_u32(ha[3], s_a), 0u, xq[w].z, xq[w].w);
                }
            }
        }
        float* base = red + wk * rpi * mstride;
        if (va) {
            if (m0 < MTE) base[ra * mstride + m0] = d[0] * e2a;
            if (m0 + 1 < MTE) base[ra * mstride + m0 + 1] = d[1] * e2b;
        }
        if (vb) {
            if (m0 < MTE) base[rb * mstride + m0] = d[2] * e2a;
            if (m0 + 1 < MTE) base[rb * mstride + m0 + 1] = d[3] * e2b;
        }
    }
}

// ------------------------------------------------------------------ item bookkeeping

struct Item {
    int group;   // dense: weight tensor (0 gate / 1 up); MoE: expert group
    int row0;
    int rows;
};

// Walks a contiguous block of items in order without per-item divisions.
struct ItemWalk {
    int group, chunk;
    __device__ __forceinline__ ItemWalk(const Params& p, int it) : group(it / p.chunks), chunk(it - (it / p.chunks) * p.chunks) {}
    __device__ __forceinline__ Item get(const Params& p) const {
        Item r;
        r.group = group;
        r.row0 = chunk * p.rpi;
        r.rows = min(p.rpi, p.N - r.row0);
        return r;
    }
    __device__ __forceinline__ void next(const Params& p) {
        if (++chunk == p.chunks) {
            chunk = 0;
            ++group;
        }
    }
};

// MoE: expert groups from the routing (same result in every CTA). A group is up to
// p.mstride slots routed to one expert; slots of one expert are served by one read.
__device__ void build_moe_tables(const Params& p, MoeTables* tab, int* scratch) {
    const int tid = threadIdx.x;
    int* ids = scratch;                       // [slots]
    int* ngr = scratch + kMaxMoeSlots;        // groups opened by slot t (leaders only)
    int* cnt = scratch + 2 * kMaxMoeSlots;    // members of leader t
    for (int t = tid; t < p.slots; t += blockDim.x) ids[t] = __ldg(p.ids + t);
    __syncthreads();
    for (int t = tid; t < p.slots; t += blockDim.x) {
        const int id = ids[t];
        const bool valid = id >= 0 && id < p.E;
        bool leader = valid;
        for (int u = 0; u < t && leader; ++u) leader = ids[u] != id;
        int c = 0;
        if (leader)
            for (int u = t; u < p.slots; ++u) c += ids[u] == id;
        cnt[t] = c;
        ngr[t] = leader ? (c + p.mstride - 1) / p.mstride : 0;
        if (!valid && blockIdx.x == 0) {
            raise_status(NVFP4_DEV_BAD_EXPERT, p.status_user);
            for (int n = 0; n < p.N; ++n) store_out(p.y, static_cast<int64_t>(t) * p.ldy + n, 0.f, p.out_bf16);
        }
    }
    __syncthreads();
    if (tid < 32) {
        // exclusive scan of ngr over slots, 8 slots per lane
        int local[8];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = tid * 8 + i;
            local[i] = t < p.slots ? ngr[t] : 0;
            sum += local[i];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (tid >= o) incl += v;
        }
        int run = incl - sum;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = tid * 8 + i;
            if (t < p.slots) ngr[t] = run;  // now: first group index of leader t
            run += local[i];
        }
        if (tid == 31) tab->n_groups = incl;
    }
    __syncthreads();
    for (int t = tid; t < p.slots; t += blockDim.x) {
        int c = cnt[t];
        if (c == 0) continue;
        const int id = ids[t];
        // members of expert id in slot order, written from member_list[first of group]
        int g = ngr[t];
        int in_group = 0;
        int pos = 0;
        // the member list of this leader occupies a contiguous run; its start is the
        // number of valid slots whose expert's leader comes before t, found by counting
        // members of earlier leaders.
        for (int u = 0; u < t; ++u) pos += cnt[u];
        for (int u = t; u < p.slots; ++u) {
            if (ids[u] != id) continue;
            if (in_group == 0) {
                tab->expert[g] = id;
                tab->first[g] = pos;
                tab->count[g] = min(p.mstride, c);
            }
            tab->member_list[pos++] = u;
            if (++in_group == p.mstride) {
                in_group = 0;
                c -= p.mstride;
                ++g;
            }
        }
    }
    __syncthreads();
}

// ------------------------------------------------------------------ the streaming kernel

__host__ __device__ constexpr int rows_per_batch(int mte) { return mte <= 2 ? 8 : 4; }
constexpr int kTileRows = 16;  // rows of one MMA tile (tensor-core path)
constexpr int kNumBars = 4 * kMaxStages + 5;

// Dispatches one item's consumer work to the tensor-core path (x staged row-scaled in f16)
// or the exact fp32 path.
template <int MTE>
__device__ __forceinline__ void compute_dispatch(bool use_mma, uint32_t wst, int wstride, uint32_t sst,
                                                 int srow_bytes, uint32_t xa, int xh_stride,
                                                 const uint16_t* const (&xrow)[8], const float* e2, int rows, int Kr,
                                                 int J, int wr, int wk, int cr, int ck, int lane, float* red, int rpi,
                                                 int mstride) {
    if (use_mma) {
        compute_item_mma<MTE>(wst, wstride, sst, srow_bytes, xa, xh_stride, e2, rows, Kr, wr, wk, cr, ck, lane, red,
                              rpi, mstride);
    } else {
        compute_item_f32<MTE, rows_per_batch(MTE)>(wst, sst, wstride, srow_bytes, xrow, rows, Kr, J, wr, wk, cr, ck,
                                                   lane, red, rpi, mstride);
    }
}

template <int MODE, int MT>
__global__ void __launch_bounds__(kThreads, 2) gemv_stream_kernel(const __grid_constant__ Params p) {
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* bars = reinterpret_cast<uint64_t*>(smem + p.bar_off);
    uint64_t* full = bars;
    uint64_t* empty = bars + kMaxStages;
    uint64_t* rfull = bars + 2 * kMaxStages;
    uint64_t* rempty = bars + 3 * kMaxStages;
    uint64_t* xready = bars + 4 * kMaxStages;
    uint64_t* xfree = bars + 4 * kMaxStages + 1;
    uint64_t* xmax = bars + 4 * kMaxStages + 2;
    uint64_t* xraw_full = bars + 4 * kMaxStages + 3;   // raw x rows landed (bulk copies)
    uint64_t* xraw_empty = bars + 4 * kMaxStages + 4;  // consumers converted them
    volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + kNumBars);
    volatile int* lossy_flag = abort_flag + 1;
    float* red_base = reinterpret_cast<float*>(smem + p.red_off);
    float* clpart = reinterpret_cast<float*>(smem + p.cl_off);
    MoeTables* tab = reinterpret_cast<MoeTables*>(smem + p.tab_off);
    float* e2 = reinterpret_cast<float*>(smem + p.misc_off);              // [8]
    uint32_t* wmax = reinterpret_cast<uint32_t*>(smem + p.misc_off) + 8;  // [kConsumerWarps][16]

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int rank = p.S > 1 ? static_cast<int>(cluster_rank()) : 0;
    const int cluster = blockIdx.x / p.S;
    const int n_clusters = gridDim.x / p.S;
    const int k0 = rank * p.Kr;
    const int NS = p.stages;

    if (threadIdx.x == 0) {
        for (int i = 0; i < NS; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], kConsumerWarps);
            mbar_init(&rfull[i], kConsumerWarps);
            mbar_init(&rempty[i], 1);
        }
        mbar_init(xready, kConsumerWarps);
        mbar_init(xfree, kConsumerWarps);
        mbar_init(xmax, kConsumerWarps);
        mbar_init(xraw_full, 1);
        mbar_init(xraw_empty, kConsumerWarps);
        *abort_flag = 0;
        *lossy_flag = 0;
        fence_barrier_init();
    }
    if constexpr (MODE == kModeMoe) {
        pdl_wait();  // the routing may come from the preceding kernel
        build_moe_tables(p, tab, reinterpret_cast<int*>(red_base));
    }
    __syncthreads();
    pdl_launch_dependents();

    // this cluster's contiguous block of items: q or q + 1 of them
    int ib, ie;
    if constexpr (MODE == kModeMoe) {
        const int items = tab->n_groups * p.chunks;
        const int q = items / n_clusters, r = items - q * n_clusters;
        ib = cluster * q + min(cluster, r);
        ie = ib + q + (cluster < r ? 1 : 0);
    } else {
        ib = cluster * p.items_q + min(cluster, p.items_r);
        ie = ib + p.items_q + (cluster < p.items_r ? 1 : 0);
    }
    const int64_t Kh = p.K / 2;
    const int64_t Ks = p.K / 16;
    const int srow_bytes = p.S == 1 ? p.K / 16 : p.Kr / 16;
    const uint32_t scale_region = static_cast<uint32_t>(p.rpi) * p.wstride;  // multiple of 64

    if (warp == kProducerWarp) {
        // ---------------- producer: TMA bulk copies of the (read-only) weights into the ring,
        // and of the raw x rows. Weights may stream before the preceding kernel has finished;
        // x is copied only after it has (pdl_wait).
        int issued = 0;
        int xkey = -1, xq = 0;  // rows whose x copy was issued; copies issued so far
        bool xfirst_pending = true;
        ItemWalk walk(p, ib);
        int slot = 0, use = 0;
        for (int it = ib; it < ie; ++it, walk.next(p), slot = slot + 1 == NS ? 0 : slot + 1, use += slot == 0) {
            const int li = it - ib;
            if (use > 0 && !mbar_wait(&empty[slot], (use - 1) & 1, p.wait_ns)) {
                *abort_flag = 1;
                if (lane == 0) raise_status(NVFP4_DEV_TIMEOUT, p.status_user);
                break;
            }
            if (*abort_flag) break;
            const Item ii = walk.get(p);
            const uint8_t* wsrc;
            const uint8_t* ssrc;
            if constexpr (MODE == kModeMoe) {
                const int64_t e = tab->expert[ii.group];
                wsrc = p.w[0] + (e * p.N + ii.row0) * Kh;
                ssrc = p.s[0] + (e * p.N + ii.row0) * Ks;
            } else {
                wsrc = p.w[ii.group] + static_cast<int64_t>(ii.row0) * Kh;
                ssrc = p.s[ii.group] + static_cast<int64_t>(ii.row0) * Ks;
            }
            uint8_t* wdst = smem + slot * p.stage_stride;
            uint8_t* sdst = wdst + scale_region;
            const uint32_t wb = p.Kr / 2;
            uint32_t sbytes_tx = 0;
            uint32_t mis = 0, head = 0, mid = 0, tail = 0;
            if (p.S > 1 || p.s_aligned) {
                sbytes_tx = static_cast<uint32_t>(ii.rows) * srow_bytes;
            } else {
                // unaligned scale range: plain copies of the head and tail bytes, TMA for the rest
                const uint32_t sbytes = static_cast<uint32_t>(ii.rows) * srow_bytes;
                mis = static_cast<uint32_t>(reinterpret_cast<uintptr_t>(ssrc) & 15);
                head = (16 - mis) & 15;
                if (head > sbytes) head = sbytes;
                mid = (sbytes - head) & ~15u;
                tail = sbytes - head - mid;
                if (lane < head) sdst[mis + lane] = ssrc[lane];
                if (lane < tail) sdst[mis + head + mid + lane] = ssrc[head + mid + lane];
                sbytes_tx = mid;
            }
            __syncwarp();  // the plain copies are ordered before the arrive below
            if (lane == 0) mbar_arrive_expect_tx(&full[slot], static_cast<uint32_t>(ii.rows) * wb + sbytes_tx);
            __syncwarp();
            if (p.S == 1) {
                // whole rows are contiguous in HBM and in the slot: one copy for the codes
                if (lane == 0) {
                    bulk_g2s(wdst, wsrc, static_cast<uint32_t>(ii.rows) * wb, &full[slot]);
                    if (p.s_aligned) bulk_g2s(sdst, ssrc, sbytes_tx, &full[slot]);
                    else if (mid) bulk_g2s(sdst + mis + head, ssrc + head, mid, &full[slot]);
                }
            } else {
                for (int r = lane; r < ii.rows; r += 32) {
                    bulk_g2s(wdst + r * p.wstride, wsrc + r * Kh + k0 / 2, wb, &full[slot]);
                    bulk_g2s(sdst + r * srow_bytes, ssrc + r * Ks + k0 / 16, srow_bytes, &full[slot]);
                }
            }
            __syncwarp();
            issued = li + 1;
            // raw x rows: dense x once, right after the first item's weights are on their way;
            // MoE each time the expert group changes, once the consumers have released the buffer
            const int key = MODE == kModeMoe ? ii.group : 0;
            const bool want_x = MODE == kModeMoe ? key != xkey : xfirst_pending;
            if (want_x) {
                if (xq > 0 && !mbar_wait(xraw_empty, (xq - 1) & 1, p.wait_ns)) {
                    *abort_flag = 1;
                    if (lane == 0) raise_status(NVFP4_DEV_TIMEOUT, p.status_user);
                    break;
                }
                if constexpr (MODE != kModeMoe) pdl_wait();  // x may come from the preceding kernel
                int nrows = MT, first = 0;
                if constexpr (MODE == kModeMoe) {
                    nrows = tab->count[key];
                    first = tab->first[key];
                }
                const uint32_t rb = static_cast<uint32_t>(p.Kr) * 2;
                if (lane == 0) mbar_arrive_expect_tx(xraw_full, static_cast<uint32_t>(nrows) * rb);
                __syncwarp();
                for (int m = lane; m < nrows; m += 32) {
                    int row = m;
                    if constexpr (MODE == kModeMoe) {
                        const int sl = tab->member_list[first + m];
                        row = p.x_per_slot ? sl : sl / p.top_k;
                    }
                    bulk_g2s(smem + p.xraw_off + m * rb, p.x + static_cast<int64_t>(row) * p.K + k0, rb, xraw_full);
                }
                __syncwarp();
                xkey = key;
                ++xq;
                xfirst_pending = false;
            }
        }
        if (xq > 0) mbar_wait(xraw_full, (xq - 1) & 1, kDrainWaitNs);
        // Every slot's latest issued copy must land before the CTA can retire, also when the
        // consumers gave up early. In a normal run these waits return at once.
        for (int li = issued - 1; li >= 0 && li >= issued - NS; --li) {
            mbar_wait(&full[li % NS], (li / NS) & 1, kDrainWaitNs);
        }
    } else if (warp == kEpilogueWarp) {
        // ---------------- epilogue: fixed-order sum over K-warps, scale, store
        int64_t local_row = 0;
        ItemWalk walk(p, ib);
        int slot = 0, use = 0;
        for (int it = ib; it < ie; ++it, walk.next(p), slot = slot + 1 == NS ? 0 : slot + 1, use += slot == 0) {
            if (!mbar_wait(&rfull[slot], use & 1, p.wait_ns)) {
                *abort_flag = 1;
                if (lane == 0) raise_status(NVFP4_DEV_TIMEOUT, p.status_user);
                break;
            }
            if (*abort_flag) break;
            const Item ii = walk.get(p);
            const float* red = red_base + slot * (p.ck * p.rpi * p.mstride);
            int mrows = MT;
            float gsc = 0.f;
            if constexpr (MODE == kModeMoe) {
                mrows = tab->count[ii.group];
                gsc = __ldg(p.g_dev + tab->expert[ii.group]);
            } else {
                gsc = p.g[ii.group];
            }
            const int total = mrows * ii.rows;
            for (int idx = lane; idx < total; idx += 32) {
                const int m = idx / ii.rows;
                const int r = idx - m * ii.rows;
                float v = 0.f;
                for (int c = 0; c < p.ck; ++c) v += red[(c * p.rpi + r) * p.mstride + m];
                if (p.S > 1) {
                    clpart[(local_row + r) * p.mstride + m] = v;
                } else if constexpr (MODE == kModeMoe) {
                    const int sl = tab->member_list[tab->first[ii.group] + m];
                    store_out(p.y, static_cast<int64_t>(sl) * p.ldy + ii.row0 + r, gsc * v, p.out_bf16);
                } else {
                    store_out(p.y, m * p.ldy + static_cast<int64_t>(ii.group) * p.N + ii.row0 + r, gsc * v, p.out_bf16);
                }
            }
            local_row += ii.rows;
            __syncwarp();
            if (lane == 0) mbar_arrive(&rempty[slot]);
        }
    } else {
        // ---------------- consumers
        const int wk = warp % p.ck;
        const int wr = warp / p.ck;
        const int ctid = threadIdx.x;  // consumer warps are 0..7
        const uint32_t xa = smem_addr(smem + p.x_off);
        const uint16_t* xrow[8];
        int cur_key = -1;
        int xr = 0, xf = 0, xm = 0, xq = 0;  // completed phases of xready / xfree / xmax / xraw_full
        bool use_mma = false;
        bool ok = true;
        if constexpr (MODE != kModeMoe) pdl_wait();  // x may come from the preceding kernel
        ItemWalk walk(p, ib);
        int slot = 0, use = 0;
        for (int it = ib; it < ie && ok; ++it, walk.next(p), slot = slot + 1 == NS ? 0 : slot + 1, use += slot == 0) {
            const Item ii = walk.get(p);
            const int key = MODE == kModeMoe ? ii.group : 0;
            if (key != cur_key) {
                // hand over the x buffer: all consumers done with the old rows, then restage
                if (cur_key >= 0) {
                    __syncwarp();
                    if (lane == 0) mbar_arrive(xfree);
                    if (!mbar_wait(xfree, xf & 1, p.wait_ns)) { ok = false; break; }
                    ++xf;
                }
                int nrows = MT;
                int first = 0;
                if constexpr (MODE == kModeMoe) {
                    nrows = tab->count[key];
                    first = tab->first[key];
                }
                const int tk = p.top_k;
                const bool per_slot = p.x_per_slot != 0;
                auto src_row = [&](int m) {
                    if constexpr (MODE == kModeMoe) {
                        const int sl = tab->member_list[first + m];
                        return per_slot ? sl : sl / tk;
                    } else {
                        return m;
                    }
                };
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    xrow[m] = p.x + static_cast<int64_t>(m < nrows ? src_row(m) : 0) * p.K + k0;
                bool lossy = true;
                if (!p.force_f32) {
                    if (!mbar_wait(xraw_full, xq & 1, p.wait_ns)) { ok = false; break; }
                    bool sok = true;
                    lossy = stage_x_mma<MT>(smem + p.xraw_off, p.Kr, nrows, smem + p.x_off, p.xh_stride, e2, wmax,
                                            xmax, xm & 1, p.wait_ns, ctid, kConsumerWarps * 32, sok);
                    ++xm;
                    if (!sok) { ok = false; break; }
                } else if (!mbar_wait(xraw_full, xq & 1, p.wait_ns)) {
                    ok = false;
                    break;
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(xraw_empty);  // the raw rows may be replaced now
                ++xq;
                if (lossy) *lossy_flag = xr + 1;
                __syncwarp();
                if (lane == 0) mbar_arrive(xready);
                if (!mbar_wait(xready, xr & 1, p.wait_ns)) { ok = false; break; }
                ++xr;
                use_mma = *lossy_flag != xr;
                if (!use_mma && !p.force_f32 && ctid == 0) atomicAdd(&g_fp32_fallbacks, 1ull);
                cur_key = key;
            }
            if (!mbar_wait(&full[slot], use & 1, p.wait_ns)) { ok = false; break; }
            if (use > 0 && !mbar_wait(&rempty[slot], (use - 1) & 1, p.wait_ns)) { ok = false; break; }
            if (*abort_flag) { ok = false; break; }

            const uint32_t wst = smem_addr(smem + slot * p.stage_stride);
            uint32_t sst = wst + scale_region;
            if (p.S == 1 && !p.s_aligned) {
                const uint8_t* ssrc;
                if constexpr (MODE == kModeMoe) {
                    ssrc = p.s[0] + (static_cast<int64_t>(tab->expert[ii.group]) * p.N + ii.row0) * Ks;
                } else {
                    ssrc = p.s[ii.group] + static_cast<int64_t>(ii.row0) * Ks;
                }
                sst += static_cast<uint32_t>(reinterpret_cast<uintptr_t>(ssrc) & 15);
            }
            float* red = red_base + slot * (p.ck * p.rpi * p.mstride);
            if constexpr (MODE == kModeMoe) {
                const int cnt = tab->count[ii.group];
                switch (cnt) {
#define NVFP4_MOE_CASE(C)                                                                                        \
    case C:                                                                                                      \
        if constexpr (C <= MT)                                                                                   \
            compute_dispatch<C>(use_mma, wst, p.wstride, sst, srow_bytes, xa, p.xh_stride, xrow, e2, ii.rows,    \
                                p.Kr, p.J, wr, wk, p.cr, p.ck, lane, red, p.rpi, p.mstride);                     \
        break;
                    NVFP4_MOE_CASE(1)
                    NVFP4_MOE_CASE(2)
                    NVFP4_MOE_CASE(3)
                    NVFP4_MOE_CASE(4)
                    NVFP4_MOE_CASE(5)
                    NVFP4_MOE_CASE(6)
                    NVFP4_MOE_CASE(7)
                    NVFP4_MOE_CASE(8)
#undef NVFP4_MOE_CASE
                    default: break;
                }
            } else {
                compute_dispatch<MT>(use_mma, wst, p.wstride, sst, srow_bytes, xa, p.xh_stride, xrow, e2, ii.rows, p.Kr,
                                     p.J, wr, wk, p.cr, p.ck, lane, red, p.rpi, p.mstride);
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(&empty[slot]);
                mbar_arrive(&rfull[slot]);
            }
        }
        if (!ok) {
            *abort_flag = 1;
            if (lane == 0) raise_status(NVFP4_DEV_TIMEOUT, p.status_user);
        }
    }

    if (p.S > 1) {
        // ---------------- cluster: sum the S partials of every row over DSMEM
        __syncwarp();
        cluster_sync_all();
        if (!*abort_flag) {
            int64_t local_row = 0;
            ItemWalk walk(p, ib);
            for (int it = ib; it < ie; ++it, walk.next(p)) {
                const Item ii = walk.get(p);
                const float gsc = p.g[ii.group];
                const int total = ii.rows * p.M;
                for (int idx = threadIdx.x; idx < total; idx += blockDim.x) {
                    const int m = idx / ii.rows;
                    const int r = idx - m * ii.rows;
                    if ((r % p.S) != rank) continue;
                    const float* mine = clpart + (local_row + r) * p.mstride + m;
                    float v = 0.f;
                    for (int c = 0; c < p.S; ++c) v += ld_cluster_f32(mine, c);
                    store_out(p.y, m * p.ldy + static_cast<int64_t>(ii.group) * p.N + ii.row0 + r, gsc * v,
                              p.out_bf16);
                }
                local_row += ii.rows;
            }
        }
        cluster_sync_all();
    }
}

// ------------------------------------------------------------------ the tile kernel

// Warp-tile GEMV (dense and gate/up, K % 256 == 0, 16-byte aligned operands). Every warp
// computes: there is no producer or epilogue warp.
//   * Work unit = one 16-row tile (the MMA's M) times one K slice. A CTA walks a contiguous
//     block of items; an item is `tpi` tiles, and each tile is shared by `ksplit` warps,
//     each owning a contiguous range of the row's TMA boxes.
//   * Each warp streams its own units through a private ring of `stages` slots. Lane 0
//     issues one 3-D TMA tensor copy for the codes (16 rows x NC 128-byte segments, 128-byte
//     swizzle) and one for the scales (16 rows x NC 16-byte segments) per slot. The rows land
//     in shared memory in the order MMA row g <-> physical row perm(g), which makes the
//     swizzled 128-bit reads of an MMA quad free of bank conflicts.
//   * Weights are requested before griddepcontrol.wait, so under programmatic dependent
//     launch they stream while the preceding kernel finishes. x is read only afterwards.
//   * x is read from global memory and staged in f16 by the warps that share a K slice, for
//     that slice only, with one power of two per row and slice (exactness is checked;
//     otherwise those warps compute in fp32 on CUDA cores).
//   * Partial sums of a tile's K slices are added in a fixed order through shared memory;
//     with ksplit == 1 each warp stores its tile directly.

namespace tk {
constexpr int kWarps = 8;
constexpr int kThreads = kWarps * 32;
constexpr int kMaxStages = 4;
constexpr int kRedFloats = kWarps * 16 * 8;  // one item's partial sums: [warp][row][m]
}  // namespace tk

struct TileParams {
    CUtensorMap wmap[2];      // codes of each group viewed as (128 B, K/256, rows)
    CUtensorMap smap[2];      // scales viewed as (16 B, K/256, rows)
    const uint16_t* x;        // bf16 bits [M, K]
    void* y;
    float g[2];
    int64_t ldy;              // y row stride in elements
    int out_bf16;
    int M, N, K;
    int tiles;                // 16-row tiles per group (fused gate/up: 2 per output tile, gate then up)
    int ksplit_log2;          // warps sharing one tile (K slices) = 1 << ksplit_log2
    int tpi;                  // tiles per item (= kWarps / ksplit)
    int ipg;                  // items per group
    int items_q, items_r;     // items per unit (a CTA, or a cluster of S CTAs): q, plus one for the first r
    int s_log2;               // CTAs per cluster S = 1 << s_log2; rank r takes the r-th of S K ranges
    int nbox;                 // TMA boxes per row
    int stages;               // ring slots per warp
    int force_f32;
    int swiglu;               // gate/up with the fused activation: tile 2j is gate tile j, 2j+1 up tile j
    float clamp;              // its clamp limit (+inf: none)
    uint32_t sstride;         // bytes between staged x rows of one K slice (64 mod 128)
    uint32_t ring_w, ring_s, x_off, red_off, cpart_off, misc_off, bar_off;  // offsets from the 1024-aligned base
    uint64_t wait_ns;
    // routed experts (MoE launches only)
    const int32_t* ids;       // expert per slot [slots]
    const float* g_dev;       // global scale per expert [E]
    int32_t* status_user;     // optional device status word
    int E, top_k, slots, x_per_slot;
    uint32_t moe_off;         // TileMoe tables
    int trace_slot;           // phase-trace launch slot (diagnostic builds only)
    // dictionary scales: smap[] views the index planes; table of E4M3 codes [32] ([E][32] MoE)
    const uint8_t* sd_dict;
    int sd_tiles;             // 16-row tiles per expert in the index plane (MoE)
    uint32_t sdtab_off;       // the pair table: 1024 f16x2 scale pairs
};

// Bytes of one ring slot's scale box: NC 16-byte rows of E4M3 codes per tile row, or (dictionary
// scales) NC 160-byte index records, padded to 128 bytes.
template <int NC, bool SD>
__host__ __device__ constexpr uint32_t scale_box_bytes() {
    return SD ? (NC * kSdRecord + 127) / 128 * 128 : NC * 256;
}

// Bytes one scale box copy delivers.
template <int NC, bool SD>
__host__ __device__ constexpr uint32_t scale_box_tx() {
    return SD ? NC * kSdRecord : NC * 256;
}

// Routed-expert groups of one launch, built by every CTA from the ids: a group is one expert
// and up to 8 of its slots (the MMA's 8 columns), groups ordered by their first slot.
constexpr int kTileMoeSlots = 32;
constexpr int kMoeWindow = 4;                 // groups a stream-K CTA may touch when slots > 32
struct TileMoe {
    int n_groups;
    int nrows;                                // x rows this CTA stages
    int g0;                                   // group of entry 0 (the arrays hold groups g0, g0 + 1, ...)
    int expert[kTileMoeSlots];
    int count[kTileMoeSlots];
    int slot[kTileMoeSlots][8];               // member slots, slot order
    int col[kTileMoeSlots][8];                // staged x row of each member
    int xrow[kTileMoeSlots][8];               // x row (global) of each member
    int rows[kTileMoeSlots];                  // global x row of each staged row
};

#ifndef NVFP4_EVICT_FIRST
#define NVFP4_EVICT_FIRST 1  // 1: weight copies carry an L2 evict-first policy (read once; vocab 0.93 -> 0.98 of the copy peak)
#endif

// An L2 policy that evicts the lines it tags first: weights are streamed once, so they should not
// push x, the expert ids or the outputs out of L2.
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const CUtensorMap* map, int c0, int c1, int c2,
                                            uint32_t bar) {
#if NVFP4_EVICT_FIRST
    const uint64_t pol = l2_evict_first_policy();
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1, {%2, %3, %4}], [%5], %6;"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(pol) : "memory");
#else
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
        ::"r"(dst), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(bar) : "memory");
#endif
}

#ifndef NVFP4_PREFETCH_TMAP
#define NVFP4_PREFETCH_TMAP 1  // 1: fetch the launch's tensor-map descriptors at kernel entry
#endif

// Starts fetching a tensor-map descriptor (kernel parameter space) into the descriptor cache, so
// the first copy that uses it does not wait for the fetch.
__device__ __forceinline__ void prefetch_tmap(const CUtensorMap* map) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ uint4 ldg128(const void* p) {
    uint4 v;
    asm volatile("ld.global.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

// The same load cached in L2 only: for data that other CTAs of the same launch wrote (the FFN's
// h), so no L1 line from before their writes can answer it.
__device__ __forceinline__ uint4 ldcg128(const void* p) {
    uint4 v;
    asm volatile("ld.global.cg.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p) : "memory");
    return v;
}

template <bool kCG>
__device__ __forceinline__ uint4 ldx128(const void* p) {
    if constexpr (kCG) return ldcg128(p);
    else return ldg128(p);
}

// Brings [p, p + bytes) into L2 (a hint: no data is returned, so it is safe even while
// another kernel may still write that memory; L2 stays coherent with those writes).
__device__ __forceinline__ void prefetch_l2_bulk(const void* p, uint32_t bytes) {
    asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

__device__ __forceinline__ void prefetch_l2(const void* p) {
    asm volatile("prefetch.global.L2 [%0];" ::"l"(p));
}

__device__ __forceinline__ void prefetch_l1(const void* p) {
    asm volatile("prefetch.global.L1 [%0];" ::"l"(p));
}

// Shared-memory row of MMA row g (0..7) for a box of NC 128-byte segments per row. The
// 128-byte swizzle XORs the 16-byte unit index with bits 7..9 of the address, i.e. with
// (row * NC + segment) & 7. The two MMA rows served by one 8-lane phase of a 128-bit load
// (g = 2p, 2p + 1) then differ in bit 2 of that value, so they hit disjoint bank halves.
template <int NC>
__host__ __device__ __forceinline__ int tile_row_perm(int g) {
    if constexpr (NC == 1) return ((g & 1) << 2) | (g >> 1);
    else if constexpr (NC == 2) return (g & 4) | ((g & 1) << 1) | ((g >> 1) & 1);
    else return g;
}

#ifndef NVFP4_STAGE_PRE
#define NVFP4_STAGE_PRE 2
#endif
#ifndef NVFP4_SK_STAGE_PRE
#define NVFP4_SK_STAGE_PRE 2  // loads in flight per lane when the stream-K form stages x (8 measured no better)
#endif
#ifndef NVFP4_DENSE_EARLY
#define NVFP4_DENSE_EARLY 4  // ring slots a dense warp requests before the dependency wait (the rest after x staging)
#endif

// Fast staging of x[:, k0 : k0 + kn] for the warps of one K slice: every bf16 value is
// converted to f16 unscaled, which is exact when it is zero or 2^-17 <= |x| < 2^16 (a bf16
// value has 8 significant bits; f16 keeps them down to its subnormal step 2^-24). One pass,
// no reduction: each lane checks its own values and the slice votes. Returns true when every
// value converted exactly (uniform over the slice's warps); otherwise the caller re-stages
// with a power-of-two scale. `vote` is gw words of shared scratch; bar_id < 0: one warp.
// after_issue() runs once the first loads are out (M > 0 or not).
template <int kPre = NVFP4_STAGE_PRE, bool kCG = false, typename F>
__device__ bool stage_x_direct(const uint16_t* __restrict__ x, const int* rowsel, int M, int K, int k0, int kn,
                               uint8_t* xs, uint32_t sstride, uint32_t* vote, int gi, int gw, int bar_id, int lane,
                               F&& after_issue) {
    const int cpr = kn >> 3;
    const int tl = gi * 32 + lane, nt = gw * 32;
    int m = 0, c = tl;
    while (c >= cpr) {
        c -= cpr;
        ++m;
    }
    uint32_t bad = 0u;
    auto convert = [&](const uint4& q, int mm, int cc) {
        const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t mag = w4[i] & 0x7fff7fffu;
            // lanes (16-bit halves) that are nonzero and below 2^-17 (0x3700), or >= 2^16 (0x4780)
            bad |= (__vcmpltu2(mag, 0x37003700u) & ~__vcmpeq2(mag, 0u)) | __vcmpgeu2(mag, 0x47804780u);
            const __half2 h = __floats2half2_rn(bf16_lo(w4[i]), bf16_hi(w4[i]));
            out[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(xs + mm * sstride + mma_x_off(cc * 8)) = make_uint4(out[0], out[1], out[2], out[3]);
    };
    auto advance = [&]() {
        c += nt;
        while (c >= cpr) {
            c -= cpr;
            ++m;
        }
    };
    // batches of kPre loads in flight, so a lane's chunks cost one L2 round trip per batch
    bool first = true;
    do {
        uint4 v[kPre];
        int mi[kPre], ci[kPre];
#pragma unroll
        for (int i = 0; i < kPre; ++i) {
            mi[i] = m;
            ci[i] = c;
            v[i] = m < M ? ldx128<kCG>(x + static_cast<int64_t>(rowsel ? rowsel[m] : m) * K + k0 + c * 8)
                         : make_uint4(0u, 0u, 0u, 0u);
            advance();
        }
        if (first) after_issue();  // the caller's own requests queue behind these loads, not in front
        first = false;
#pragma unroll
        for (int i = 0; i < kPre; ++i)
            if (mi[i] < M) convert(v[i], mi[i], ci[i]);
    } while (m < M);
    bool ok = !__any_sync(0xffffffffu, bad != 0u);
    if (bar_id >= 0) {
        if (lane == 0) vote[gi] = ok ? 1u : 0u;
        named_bar_sync(bar_id, gw * 32);
        for (int w = 0; w < gw; ++w) ok = ok && vote[w] != 0u;
    } else {
        __syncwarp();
    }
    return ok;
}

#ifndef NVFP4_STAGE_BULK
#define NVFP4_STAGE_BULK 0  // 1: x arrives by bulk copies and is converted in place (correct, but measured slower)
#endif

// stage_x_direct with the slice's rows brought in by bulk copies: lane 0 of the slice's first
// warp copies each row's K range (raw bf16, kn * 2 bytes) to its place in the staged buffer,
// completing on the mbarrier `bar` (8 bytes of shared scratch, initialised here). Every
// 256-byte block (128 elements) is then converted in place by half a warp: its sixteen
// 16-byte chunks, raw chunk 4t + q holding elements 32t + 8q .. + 7, move to position 4q + t
// (the mma_x_off order) as f16, with the same exactness check and slice vote. One L2 round
// trip for the whole slice instead of one per batch of loads. A wait that runs out (budget)
// sets NVFP4_DEV_TIMEOUT, drains the copy and reports the slice inexact, so the caller
// re-stages it from global memory. Needs 16-byte aligned x rows and k0 and kn multiples of 128.
// Iterations of stage_x_bulk's in-place conversion loop for warp gi of gw sharing nblk 256-byte
// blocks (two per warp and iteration, one per half-warp). It depends on no lane and no x value:
// the loop body holds a __syncwarp, so every lane of the warp must run the same count.
__host__ __device__ __forceinline__ int bulk_convert_trips(int gi, int gw, int nblk) {
    return gi * 2 < nblk ? (nblk - gi * 2 + gw * 2 - 1) / (gw * 2) : 0;
}

__device__ bool stage_x_bulk(const uint16_t* __restrict__ x, const int* rowsel, int M, int K, int k0, int kn,
                             uint8_t* xs, uint32_t sstride, uint32_t* vote, uint64_t* bar, int gi, int gw,
                             int bar_id, int lane, uint64_t budget) {
    if (gi == 0 && lane == 0) {
        mbar_init(bar, 1);
        fence_barrier_init();
        mbar_arrive_expect_tx(bar, static_cast<uint32_t>(M) * static_cast<uint32_t>(kn) * 2u);
        for (int m = 0; m < M; ++m)
            bulk_g2s(xs + m * sstride, x + static_cast<int64_t>(rowsel ? rowsel[m] : m) * K + k0,
                     static_cast<uint32_t>(kn) * 2u, bar);
    }
    if (bar_id >= 0) named_bar_sync(bar_id, gw * 32);  // the barrier is initialised before any wait
    else __syncwarp();
    uint32_t bad = 0u;
    bool landed = true;  // warp-uniform
    if (!__all_sync(0xffffffffu, budget != 0 && mbar_wait(bar, 0u, budget))) {
        if (lane == 0) {
            raise_status(NVFP4_DEV_TIMEOUT, nullptr);
            mbar_wait(bar, 0u, kDrainWaitNs);  // the copy must not land after the re-staging
        }
        __syncwarp();
        bad = 1u;
        landed = false;
    }
    const int bpr = kn >> 7;  // 128-element blocks per row
    const int nblk = M * bpr;
    const int half = lane >> 4, pos = lane & 15;
    const int t = pos >> 2, q = pos & 3;
    // the trip count must not depend on the lane: the loop body holds a __syncwarp
    const int trips = landed ? bulk_convert_trips(gi, gw, nblk) : 0;
    for (int it = 0; it < trips; ++it) {
        const int b = gi * 2 + it * gw * 2 + half;
        uint8_t* blk = nullptr;
        uint4 v = make_uint4(0u, 0u, 0u, 0u);
        if (b < nblk) {
            const int m = b / bpr;
            blk = xs + m * sstride + (b - m * bpr) * 256;
            v = *reinterpret_cast<const uint4*>(blk + pos * 16);
        }
        __syncwarp();  // every chunk of the block is read before any is overwritten
        if (b < nblk) {
            const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
            uint32_t out[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t mag = w4[i] & 0x7fff7fffu;
                bad |= (__vcmpltu2(mag, 0x37003700u) & ~__vcmpeq2(mag, 0u)) | __vcmpgeu2(mag, 0x47804780u);
                const __half2 h = __floats2half2_rn(bf16_lo(w4[i]), bf16_hi(w4[i]));
                out[i] = *reinterpret_cast<const uint32_t*>(&h);
            }
            *reinterpret_cast<uint4*>(blk + (q * 4 + t) * 16) = make_uint4(out[0], out[1], out[2], out[3]);
        }
    }
    bool ok = !__any_sync(0xffffffffu, bad != 0u);
    if (bar_id >= 0) {
        if (lane == 0) vote[gi] = ok ? 1u : 0u;
        named_bar_sync(bar_id, gw * 32);
        for (int w = 0; w < gw; ++w) ok = ok && vote[w] != 0u;
    } else {
        __syncwarp();
    }
    return ok;
}

// Stages x[:, k0 : k0 + kn] for the warps of one K slice (gw warps; this one is number gi
// of them) in f16 for the tensor cores: rows `sstride` bytes apart at xs, elements at
// mma_x_off. The slice gets one power of two, x' = x * 2^-E with its largest |x| in
// [2^15, 2^16), and *e2 = 2^E. Exact for every value at most 2^32 below that largest one;
// a slice holding a smaller nonzero value, Inf or NaN is reported lossy
// and its warps compute in fp32 instead. Because each slice's partial sums are multiplied by
// its own e2 before slices are added, slices need no common scale and no CTA-wide step.
// The slice's rows are walked as one flat sequence of 16-byte chunks, loaded kPre at a time
// per lane; the first kPre are kept in registers for the conversion. Returns (uniform over
// the slice's warps) the lossy flag. bar_id < 0: a single warp (no named barrier).
template <bool kCG = false>
__device__ bool stage_x_slice(const uint16_t* __restrict__ x, const int* rowsel, int M, int K, int k0, int kn,
                              uint8_t* xs, uint32_t sstride, float* e2, uint32_t* gmax, int gi, int gw, int bar_id,
                              int lane) {
    constexpr int kPre = NVFP4_STAGE_PRE;
    const int cpr = kn >> 3;                      // 16-byte chunks per row of the slice
    const int tl = gi * 32 + lane, nt = gw * 32;  // this lane among the slice's lanes
    int m0 = 0, c0 = tl;                          // flat chunk tl as (row, chunk)
    while (c0 >= cpr) {
        c0 -= cpr;
        ++m0;
    }
    auto advance = [&](int& m, int& c) {
        c += nt;
        while (c >= cpr) {
            c -= cpr;
            ++m;
        }
    };
    uint4 v[kPre];
    uint32_t mx = 0u, mn = 0x7fff7fffu;
    auto scan = [&](const uint4& q) {
        const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t mag = w4[i] & 0x7fff7fffu;
            mx = __vmaxu2(mx, mag);
            mn = __vminu2(mn, mag | (__vcmpeq2(mag, 0u) & 0x7fff7fffu));
        }
    };
    {
        int m = m0, c = c0;
#pragma unroll
        for (int i = 0; i < kPre; ++i) {
            v[i] = m < M ? ldx128<kCG>(x + static_cast<int64_t>(rowsel ? rowsel[m] : m) * K + k0 + c * 8)
                         : make_uint4(0u, 0u, 0u, 0u);
            advance(m, c);
        }
#pragma unroll
        for (int i = 0; i < kPre; ++i) scan(v[i]);  // zero padding does not move max or min-nonzero
        while (m < M) {  // the rest in batches of kPre loads in flight
            uint4 u[kPre];
#pragma unroll
            for (int i = 0; i < kPre; ++i) {
                u[i] = m < M ? ldx128<kCG>(x + static_cast<int64_t>(rowsel ? rowsel[m] : m) * K + k0 + c * 8)
                             : make_uint4(0u, 0u, 0u, 0u);
                advance(m, c);
            }
#pragma unroll
            for (int i = 0; i < kPre; ++i) scan(u[i]);
        }
    }
    uint32_t a = max(mx & 0xffffu, mx >> 16), z = min(mn & 0xffffu, mn >> 16);
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
        a = max(a, __shfl_xor_sync(0xffffffffu, a, o));
        z = min(z, __shfl_xor_sync(0xffffffffu, z, o));
    }
    if (gw > 1) {
        if (lane == 0) {
            gmax[gi] = a;
            gmax[8 + gi] = z;
        }
        named_bar_sync(bar_id, gw * 32);
        for (int w = 0; w < gw; ++w) {
            a = max(a, gmax[w]);
            z = min(z, gmax[8 + w]);
        }
    }
    bool lossy = false;
    int e_max;
    if (a >= 0x7f80u || a == 0) {
        e_max = 12;                        // Inf/NaN (reported as lossy) or an all-zero slice
        lossy = a >= 0x7f80u;
    } else if ((a >> 7) == 0) {
        e_max = (31 - __clz(a)) - 133;     // bf16 subnormal: mant * 2^-133
    } else {
        e_max = static_cast<int>(a >> 7) - 127;
    }
    // largest |x'| in [2^15, 2^16): every bf16 value there (<= 65280) is an f16. Down to 2^-17
    // a bf16 value's last bit is a multiple of 2^-24, the f16 subnormal step, so it is exact too
    const int E = e_max - 15;
    const int tb = E - 17 + 127;           // smallest certainly exact magnitude 2^(E - 17), as bf16 bits
    const uint32_t thresh = tb >= 1 ? static_cast<uint32_t>(tb) << 7 : 0x80u;
    lossy |= z != 0x7fffu && z < thresh;
    if (gi == 0 && lane == 0) *e2 = pow2f(E);
    const int a2 = min(-E, 127);
    const float sa = pow2f(a2), sb = pow2f(-E - a2);  // sb == 1 unless the slice is tiny
    auto store = [&](const uint4& q, int m, int c) {
        const uint32_t w4[4] = {q.x, q.y, q.z, q.w};
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 h = __floats2half2_rn(bf16_lo(w4[i]) * sa * sb, bf16_hi(w4[i]) * sa * sb);
            out[i] = *reinterpret_cast<const uint32_t*>(&h);
        }
        *reinterpret_cast<uint4*>(xs + m * sstride + mma_x_off(c * 8)) = make_uint4(out[0], out[1], out[2], out[3]);
    };
    {
        int m = m0, c = c0;
#pragma unroll
        for (int i = 0; i < kPre; ++i) {
            if (m < M) store(v[i], m, c);
            advance(m, c);
        }
        while (m < M) {
            uint4 u[kPre];
            int mi[kPre], ci[kPre];
#pragma unroll
            for (int i = 0; i < kPre; ++i) {
                mi[i] = m;
                ci[i] = c;
                u[i] = m < M ? ldx128<kCG>(x + static_cast<int64_t>(rowsel ? rowsel[m] : m) * K + k0 + c * 8)
                             : make_uint4(0u, 0u, 0u, 0u);
                advance(m, c);
            }
#pragma unroll
            for (int i = 0; i < kPre; ++i)
                if (mi[i] < M) store(u[i], mi[i], ci[i]);
        }
    }
    if (bar_id >= 0) named_bar_sync(bar_id, gw * 32);
    else __syncwarp();
    return lossy;
}

// One ring slot on the tensor cores: NC segments x 2 steps of 128 elements. Lane (g, t)
// takes the 32 codes 32t .. 32t + 31 of each step for its rows ra = perm(g), rb = ra + 8
// (see compute_item_mma for the k permutation shared with the staged x; xa points at this
// lane's x row, `chunk0` is the slot's first 128-element chunk within the staged slice).
// Several accumulator sets (kTileChains) shorten the MMA dependency chain.
#ifndef NVFP4_TILE_CHAINS
#define NVFP4_TILE_CHAINS 4
#endif
constexpr int kTileChains = NVFP4_TILE_CHAINS;  // independent MMA accumulator chains per warp

__device__ __forceinline__ uint32_t lds32(uint32_t a) {
    uint32_t v;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(v) : "r"(a));
    return v;
}

// The f16x2 scales of blocks 8h + 2t and 8h + 2t + 1 (low half first) of tile row `row` in
// segment c of a ring slot's scale box: two E4M3 codes, or (SD) the 10-bit pair of dictionary
// indices at bit 5q, q = 16 row + 8h + 2t, looked up in the pair table at `tab`.
template <int NC, bool SD>
__device__ __forceinline__ uint32_t slot_scale2(uint32_t sst, int c, int row, int h, int t, uint32_t tab) {
    if constexpr (SD) {
        const uint32_t bit = static_cast<uint32_t>(row * 80 + h * 40 + t * 10);
        const uint32_t a = sst + c * kSdRecord + ((bit >> 5) << 2);
        const uint32_t pair = __funnelshift_r(lds32(a), lds32(a + 4), bit & 31u) & 0x3ffu;
        return lds32(tab + pair * 4);
    } else {
        return cvt_e4m3x2(lds16(sst + (row * NC + c) * 16 + h * 8 + 2 * t));
    }
}

// Fills the pair table at tab (1024 words): entry i1 * 32 + i0 holds the f16x2 of
// (E4M3(dict[i0]), E4M3(dict[i1])). Called by all `nthreads` threads; the caller synchronises.
__device__ __forceinline__ void build_pair_table(uint32_t* tab, const uint8_t* dict, int tid, int nthreads) {
    for (int e = tid; e < kSdPairs; e += nthreads)
        tab[e] = cvt_e4m3x2(static_cast<uint16_t>(__ldg(dict + (e & 31)) | (__ldg(dict + (e >> 5)) << 8)));
}

template <int NC, bool SD = false>
__device__ __forceinline__ void tile_slot_mma(uint32_t wst, uint32_t sst, uint32_t xa, int chunk0, int ra, int t,
                                              float (&dd)[kTileChains][4], uint32_t tab = 0) {
    const int rb = ra + 8;
#pragma unroll
    for (int c = 0; c < NC; ++c) {
        const int la = ra * NC + c, lb = rb * NC + c;
#pragma unroll
        for (int h = 0; h < 2; ++h) {
            const int u = h * 4 + t;
            const uint4 wa = lds128(wst + la * 128 + ((u ^ (la & 7)) << 4));
            const uint4 wb = lds128(wst + lb * 128 + ((u ^ (lb & 7)) << 4));
            const uint32_t sa = slot_scale2<NC, SD>(sst, c, ra, h, t, tab);
            const uint32_t sb = slot_scale2<NC, SD>(sst, c, rb, h, t, tab);
            const int chunk = chunk0 + c * 2 + h;
            uint4 xq[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) xq[q] = lds128(xa + chunk * 256 + ((q * 4 + t) << 4));
            const uint32_t sa0 = prmt(sa, 0x1010u), sa1 = prmt(sa, 0x3232u);
            const uint32_t sb0 = prmt(sb, 0x1010u), sb1 = prmt(sb, 0x3232u);
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                uint32_t ha[4], hb[4];
                cvt_e2m1x8(w == 0 ? wa.x : (w == 1 ? wa.y : (w == 2 ? wa.z : wa.w)), ha);
                cvt_e2m1x8(w == 0 ? wb.x : (w == 1 ? wb.y : (w == 2 ? wb.z : wb.w)), hb);
                const uint32_t s_a = w < 2 ? sa0 : sa1, s_b = w < 2 ? sb0 : sb1;
                mma_16816(dd[(2 * w) % kTileChains], hmul2_u32(ha[0], s_a), hmul2_u32(hb[0], s_b),
                          hmul2_u32(ha[1], s_a), hmul2_u32(hb[1], s_b), xq[w].x, xq[w].y);
                mma_16816(dd[(2 * w + 1) % kTileChains], hmul2_u32(ha[2], s_a), hmul2_u32(hb[2], s_b),
                          hmul2_u32(ha[3], s_a), hmul2_u32(hb[3], s_b), xq[w].z, xq[w].w);
            }
        }
    }
}

// The same slot in exact fp32 on the CUDA cores, x read from global memory (bf16): column m
// uses x row xrow[m] (row m when xrow is null). acc[r][m] collects rows ra (r = 0) and
// rb (r = 1) for column m, over this lane's 32-code pieces.
template <int NC, bool SD = false, bool kCG = false>
__device__ __noinline__ void tile_slot_f32(uint32_t wst, uint32_t sst, const uint16_t* __restrict__ x,
                                           const int* xrow, int K, int M, int kseg0, int ra, int t, float* acc,
                                           uint32_t tab = 0) {
    const int rb = ra + 8;
    for (int c = 0; c < NC; ++c) {
        const int la = ra * NC + c, lb = rb * NC + c;
        for (int h = 0; h < 2; ++h) {
            const int u = h * 4 + t;
            const uint4 wv[2] = {lds128(wst + la * 128 + ((u ^ (la & 7)) << 4)),
                                 lds128(wst + lb * 128 + ((u ^ (lb & 7)) << 4))};
            const uint32_t sh[2] = {slot_scale2<NC, SD>(sst, c, ra, h, t, tab),
                                    slot_scale2<NC, SD>(sst, c, rb, h, t, tab)};
            const int k0 = ((kseg0 + c) * 2 + h) * 128 + 32 * t;
            for (int w = 0; w < 4; ++w) {
                for (int m = 0; m < M; ++m) {
                    const uint4 xv = ldx128<kCG>(x + static_cast<int64_t>(xrow ? xrow[m] : m) * K + k0 + w * 8);
                    const uint32_t xw[4] = {xv.x, xv.y, xv.z, xv.w};
                    for (int r = 0; r < 2; ++r) {
                        const uint32_t word = w == 0 ? wv[r].x : (w == 1 ? wv[r].y : (w == 2 ? wv[r].z : wv[r].w));
                        const uint16_t sc = static_cast<uint16_t>(w < 2 ? (sh[r] & 0xffffu) : (sh[r] >> 16));
                        uint32_t hq[4];
                        cvt_e2m1x8(word, hq);
                        float a = acc[r * 8 + m];
                        for (int i = 0; i < 4; ++i) {
                            const float2 q = widen_scaled(hq[i], sc);
                            a = fmaf(q.x, bf16_lo(xw[i]), a);
                            a = fmaf(q.y, bf16_hi(xw[i]), a);
                        }
                        acc[r * 8 + m] = a;
                    }
                }
            }
        }
    }
}

// Position in a CTA's block of items, walked without divisions.
struct TileItemWalk {
    int grp, t;  // group (dense: 0 gate / 1 up; MoE: expert group) and item index within it
    __host__ __device__ __forceinline__ void next(int ipg) {
        if (++t == ipg) {
            t = 0;
            ++grp;
        }
    }
};

// Builds the routed-expert groups (warp 0; slots <= 32). Slot s with expert e joins the
// group that holds e's slots of ranks 8q .. 8q + 7, where its rank counts the earlier slots
// routed to e; groups are numbered in the order of their first slots. Invalid ids form no
// group: CTA 0 zeroes their outputs and flags them.
__device__ void tile_moe_groups(const TileParams& p, TileMoe* tab, int lane) {
    const int s = lane;
    const int id = s < p.slots ? __ldg(p.ids + s) : -1;
    const bool valid = s < p.slots && id >= 0 && id < p.E;
    const uint32_t same = __match_any_sync(0xffffffffu, valid ? id : -1 - lane);  // invalid lanes stay alone
    const uint32_t lower = (1u << lane) - 1u;
    const int rank = __popc(same & lower);
    const bool leader = valid && (rank & 7) == 0;
    const uint32_t leaders = __ballot_sync(0xffffffffu, leader);
    if (valid) {
        uint32_t rest = same;  // drop the members ranked below this group's first one
        for (int i = 0; i < (rank & ~7); ++i) rest &= rest - 1u;
        const int lead_lane = __ffs(rest) - 1;
        const int g = __popc(leaders & ((1u << lead_lane) - 1u));
        const int j = rank & 7;
        tab->slot[g][j] = s;
        tab->xrow[g][j] = p.x_per_slot ? s : s / p.top_k;
        if (j == 0) {
            tab->expert[g] = id;
            tab->count[g] = min(8, __popc(same) - rank);
        }
    }
    if (lane == 0) {
        tab->n_groups = __popc(leaders);
        tab->g0 = 0;
    }
    if (!valid && s < p.slots && blockIdx.x == 0) {
        raise_status(NVFP4_DEV_BAD_EXPERT, p.status_user);
        for (int n = 0; n < p.N; ++n) store_out(p.y, static_cast<int64_t>(s) * p.N + n, 0.f, p.out_bf16);
    }
    __syncwarp();
}

// The x rows that groups [g0, g1] need, staged in increasing row order (at most 32 rows).
// Routed-expert groups of a stream-K launch with more than 32 slots (up to kMaxMoeSlots), built
// by all threads: a sort of the (expert, slot) keys (moe_rank_by_sort) gives each slot its rank
// among the earlier slots of its expert, its expert's slot count and first slot (the leader); the
// expert's slots form groups of up to 8 in slot order, numbered from ngr[leader], leaders in slot
// order. Scratch: kMoeScratchInts ints (10.1 KB) at the start of the x region. Invalid ids form no
// group: CTA 0 zeroes their outputs and flags them.
// scratch: ids, rank, cnt, lead, ngr (5 x kMaxMoeSlots ints), two buffers of sort keys (2 x
// kMaxMoeSlots 64-bit words), the run lengths (kMaxMoeSlots ints) and the warps' scan tops (32 ints)
constexpr int kMoeScratchInts = 5 * kMaxMoeSlots + 4 * kMaxMoeSlots + kMaxMoeSlots + 32;
static_assert(kMaxMoeSlots == tk::kThreads, "the group builder sorts one slot per thread");

// Rank, expert count, leader and group count of every slot, by sorting (expert, slot) keys: after
// a bitonic sort of the kMaxMoeSlots keys (one per thread), the slots of an expert form a run in
// slot order, so a slot's rank is its distance from the run's start, its count the run's length
// and its leader the slot at the run's start. Invalid ids (negative in `ids`) and padding sort
// after every expert and form no run. All threads; ends with __syncthreads.
__device__ void moe_rank_by_sort(const int* ids, int nslots, int* rank, int* cnt, int* lead, int* ngr,
                                 unsigned long long* keys, int* runs, int* wtop, int tid) {
    const int id0 = tid < nslots ? ids[tid] : -1;
    unsigned long long key = (id0 >= 0 ? static_cast<unsigned long long>(static_cast<uint32_t>(id0)) << 32
                                       : 0xffffffffull << 32) | static_cast<uint32_t>(tid);
    // bitonic sort, one key per thread: partners within a warp swap through shuffles; partners
    // 32 or more positions apart through two alternating shared buffers (one barrier per stage)
    int buf = 0;
    for (int k = 2; k <= kMaxMoeSlots; k <<= 1) {
        for (int j = k >> 1; j > 0; j >>= 1) {
            unsigned long long other;
            if (j >= 32) {
                unsigned long long* b = keys + buf * kMaxMoeSlots;
                b[tid] = key;
                __syncthreads();
                other = b[tid ^ j];
                buf ^= 1;
            } else {
                const uint32_t lo = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(key), j);
                const uint32_t hw = __shfl_xor_sync(0xffffffffu, static_cast<uint32_t>(key >> 32), j);
                other = (static_cast<unsigned long long>(hw) << 32) | lo;
            }
            // the lower position of an ascending pair (bit k of the position clear) keeps the
            // smaller key, of a descending pair the larger
            const bool keep_min = ((tid & j) == 0) == ((tid & k) == 0);
            key = keep_min ? (key < other ? key : other) : (key > other ? key : other);
        }
    }
    keys += buf * kMaxMoeSlots;  // the buffer the last shared stage did not use
    keys[tid] = key;
    __syncthreads();
    const uint32_t hi = static_cast<uint32_t>(key >> 32);
    const bool valid = hi != 0xffffffffu;
    const bool start = tid == 0 || static_cast<uint32_t>(keys[tid - 1] >> 32) != hi;
    const bool last = tid == kMaxMoeSlots - 1 || static_cast<uint32_t>(keys[tid + 1] >> 32) != hi;
    // the start of every position's run: an inclusive max-scan of (start ? position : 0)
    int v = start ? tid : 0;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int u = __shfl_up_sync(0xffffffffu, v, o);
        if ((tid & 31) >= o) v = max(v, u);
    }
    if ((tid & 31) == 31) wtop[tid >> 5] = v;
    __syncthreads();
    for (int w = 0; w < (tid >> 5); ++w) v = max(v, wtop[w]);
    if (last) runs[v] = tid - v + 1;  // the run's length, at its start
    __syncthreads();
    const int slot = static_cast<int>(static_cast<uint32_t>(key));
    if (slot < nslots) {
        const int r = valid ? tid - v : 0;
        const int c = valid ? runs[v] : 0;
        rank[slot] = r;
        cnt[slot] = c;
        lead[slot] = valid ? static_cast<int>(static_cast<uint32_t>(keys[v])) : slot;
        ngr[slot] = valid && r == 0 ? (c + 7) / 8 : 0;
    }
    __syncthreads();
}

__device__ void tile_moe_groups_big(const TileParams& p, TileMoe* tab, int* scratch, int tid) {
    int* ids = scratch;
    int* rank = scratch + kMaxMoeSlots;
    int* cnt = scratch + 2 * kMaxMoeSlots;
    int* lead = scratch + 3 * kMaxMoeSlots;
    int* ngr = scratch + 4 * kMaxMoeSlots;
    for (int t = tid; t < kMaxMoeSlots; t += tk::kThreads) {
        int v = -2 - t;  // past the slots: matches nothing
        if (t < p.slots) {
            const int id = __ldg(p.ids + t);
            v = (id >= 0 && id < p.E) ? id : -2 - t;
            if (!(id >= 0 && id < p.E) && blockIdx.x == 0) {
                raise_status(NVFP4_DEV_BAD_EXPERT, p.status_user);
                for (int n = 0; n < p.N; ++n) store_out(p.y, static_cast<int64_t>(t) * p.N + n, 0.f, p.out_bf16);
            }
        }
        ids[t] = v;
    }
    __syncthreads();
    if (tid == 0) trace_word(p.trace_slot, 38, static_cast<unsigned long long>(clock64()));
    moe_rank_by_sort(ids, p.slots, rank, cnt, lead, ngr, reinterpret_cast<unsigned long long*>(scratch + 5 * kMaxMoeSlots),
                     scratch + 9 * kMaxMoeSlots, scratch + 10 * kMaxMoeSlots, tid);
    if (tid == 0) trace_word(p.trace_slot, 39, static_cast<unsigned long long>(clock64()));
    if (tid < 32) {
        // exclusive scan of the group counts over slots, 8 slots per lane
        int local[8];
        int sum = 0;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = tid * 8 + i;
            local[i] = t < p.slots ? ngr[t] : 0;
            sum += local[i];
        }
        int incl = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, incl, o);
            if (tid >= o) incl += v;
        }
        int run = incl - sum;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            const int t = tid * 8 + i;
            if (t < p.slots) ngr[t] = run;  // now: the first group of the expert that t leads
            run += local[i];
        }
        if (tid == 31) tab->n_groups = incl;
    }
    __syncthreads();
}

// The groups g_lo .. g_hi (at most kMoeWindow; none when g_lo > g_hi) of the CTA's job range from
// tile_moe_groups_big's scratch into tab (entry g - g_lo), then their x rows, distinct and in
// increasing order, and each member's staged column. All threads; ends with __syncthreads.
__device__ void tile_moe_window(const TileParams& p, TileMoe* tab, const int* scratch, int g_lo, int g_hi, int tid) {
    const int* ids = scratch;
    const int* rank = scratch + kMaxMoeSlots;
    const int* cnt = scratch + 2 * kMaxMoeSlots;
    const int* lead = scratch + 3 * kMaxMoeSlots;
    const int* ngr = scratch + 4 * kMaxMoeSlots;
    if (g_hi - g_lo + 1 > kMoeWindow) {  // the planner bounds the span: flag it, keep in bounds
        if (tid == 0) raise_status(NVFP4_DEV_INTERNAL, p.status_user);
        g_hi = g_lo + kMoeWindow - 1;
    }
    if (tid == 0) tab->g0 = g_lo;
    for (int u = tid; u < p.slots; u += tk::kThreads) {
        if (ids[u] < 0) continue;  // invalid id: no group
        const int r = rank[u];
        const int g = ngr[lead[u]] + (r >> 3), j = r & 7;
        if (g < g_lo || g > g_hi) continue;
        const int lg = g - g_lo;
        tab->slot[lg][j] = u;
        tab->xrow[lg][j] = p.x_per_slot ? u : u / p.top_k;
        if (j == 0) {
            tab->expert[lg] = ids[u];
            tab->count[lg] = min(8, cnt[u] - r);
        }
    }
    __syncthreads();
    if (tid < 32) {
        // lane m holds member m % 8 of window entry m / 8; a row is staged once, at the
        // position given by the number of distinct rows below it
        const int ng = g_hi - g_lo + 1;
        const int lg = tid >> 3, j = tid & 7;
        const bool has = lg < ng && j < tab->count[lg];
        const int r = has ? tab->xrow[lg][j] : 0x7fffffff;
        const uint32_t same = __match_any_sync(0xffffffffu, r);
        const bool first = has && (__ffs(same) - 1) == tid;
        const uint32_t firsts = __ballot_sync(0xffffffffu, first);
        int below = 0;
        for (int l = 0; l < 32; ++l) {
            const int v = __shfl_sync(0xffffffffu, r, l);
            below += static_cast<int>((firsts >> l) & 1u) & static_cast<int>(v < r);
        }
        if (first) tab->rows[below] = r;
        if (has) tab->col[lg][j] = below;
        if (tid == 0) tab->nrows = __popc(firsts);
    }
    __syncthreads();
}

__device__ void tile_moe_rows(const TileParams& p, TileMoe* tab, int g0, int g1, int lane) {
    // lane l takes member l % 8 of group base + l / 8: four groups per pass, one pass for the
    // usual window (a serial scan of the members took about 0.6 us of the launch's set-up)
    uint32_t want = 0u;
    for (int base = g0; base <= g1; base += 4) {
        const int g = base + (lane >> 3), j = lane & 7;
        const bool has = g <= g1 && j < tab->count[g];
        want |= __reduce_or_sync(0xffffffffu, has ? 1u << tab->xrow[g][j] : 0u);
    }
    if (lane == 0) tab->nrows = __popc(want);
    if ((want >> lane) & 1u) tab->rows[__popc(want & ((1u << lane) - 1u))] = lane;
    for (int base = g0; base <= g1; base += 4) {
        const int g = base + (lane >> 3), j = lane & 7;
        if (g <= g1 && j < tab->count[g]) tab->col[g][j] = __popc(want & ((1u << tab->xrow[g][j]) - 1u));
    }
    __syncwarp();
}

template <int NC, bool MOE, bool SWI = false, bool SD = false>
__global__ void __launch_bounds__(tk::kThreads, 2) gemv_tile_kernel(const __grid_constant__ TileParams p) {
    extern __shared__ uint8_t smem_raw[];
    constexpr uint32_t kWBox = NC * 2048;  // 16 rows x NC x 128 B
    constexpr uint32_t kSBox = scale_box_bytes<NC, SD>();  // 16 rows x NC x 16 B, or NC index records
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t = lane & 3;
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* const sbase = smem_raw + (base - raw_base);
    const int stages = p.stages;
    uint64_t* const bars = reinterpret_cast<uint64_t*>(sbase + p.bar_off) + warp * tk::kMaxStages;
    const uint32_t ring_w = base + p.ring_w + static_cast<uint32_t>(warp * stages) * kWBox;
    const uint32_t ring_s = base + p.ring_s + static_cast<uint32_t>(warp * stages) * kSBox;
    TileMoe* const tab = reinterpret_cast<TileMoe*>(sbase + p.moe_off);
    trace_begin(tid);
    if (tid == 0) trace_phase(p.trace_slot, 0);
    if (NVFP4_PREFETCH_TMAP && warp == 0 && lane < 4) prefetch_tmap(lane < 2 ? &p.wmap[lane] : &p.smap[lane - 2]);

    const int S = 1 << p.s_log2;
    const int rank = S > 1 ? static_cast<int>(cluster_rank()) : 0;
    const int unit = blockIdx.x >> p.s_log2, units = gridDim.x >> p.s_log2;
    const int c_lo = (rank * p.nbox) >> p.s_log2, c_n = (((rank + 1) * p.nbox) >> p.s_log2) - c_lo;
    const int ksplit = 1 << p.ksplit_log2;
    const int kslice = warp & (ksplit - 1), tin = warp >> p.ksplit_log2;
    const int b_lo = c_lo + ((kslice * c_n) >> p.ksplit_log2), b_hi = c_lo + (((kslice + 1) * c_n) >> p.ksplit_log2);
    const int nb = b_hi - b_lo;

    if (lane == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncwarp();
    if (tid == 0) trace_word(p.trace_slot, 32, static_cast<unsigned long long>(clock64()));

    // this unit's items: a balanced contiguous block (MoE: counted once the groups are known)
    int ib = 0, ie = 0;
    auto unit_range = [&](int items) {
        const int q = items / units, r = items - q * units;
        ib = unit * q + min(unit, r);
        ie = ib + q + (unit < r ? 1 : 0);
    };
    if constexpr (!MOE) unit_range(p.items_q * units + p.items_r);
    TileItemWalk first{0, 0};
    auto set_first = [&]() {
        first.grp = ib / p.ipg;
        first.t = ib - first.grp * p.ipg;
    };
    if constexpr (!MOE) set_first();

    // issue cursor (lane 0): the next (item, box) of this warp's units
    TileItemWalk iw = first;
    int iss_left = 0, iss_box = 0;
    uint32_t issued = 0, consumed = 0;
    // ring positions kept incrementally (the ring depth is a launch parameter: no divisions)
    uint32_t iss_st = 0, cons_st = 0, cons_ph = 0;
    auto cons_advance = [&]() {
        ++consumed;
        if (++cons_st == static_cast<uint32_t>(stages)) {
            cons_st = 0;
            cons_ph ^= 1u;
        }
    };
    auto issue_next = [&]() {
        while (iss_left > 0 && (iss_box >= nb || iw.t * p.tpi + tin >= p.tiles)) {
            iw.next(p.ipg);
            --iss_left;
            iss_box = 0;
        }
        if (iss_left <= 0) return;
        const uint32_t st = iss_st;
        if (++iss_st == static_cast<uint32_t>(stages)) iss_st = 0;
        const uint32_t bar = smem_addr(&bars[st]);
        mbar_arrive_expect_tx(&bars[st], kWBox + scale_box_tx<NC, SD>());
        const int seg = (b_lo + iss_box) * NC;
        int row0 = (iw.t * p.tpi + tin) * 16;
        int map = iw.grp;
        if constexpr (SWI) {
            map = (iw.t * p.tpi + tin) & 1;  // tiles alternate gate, up
            row0 = ((iw.t * p.tpi + tin) >> 1) * 16;
        }
        if constexpr (MOE) {
            row0 += tab->expert[iw.grp] * p.N;  // experts' rows are back to back
            map = 0;
        }
        tma_load_3d(ring_w + st * kWBox, &p.wmap[map], 0, seg, row0, bar);
        tma_load_3d(ring_s + st * kSBox, &p.smap[map], 0, seg, SD ? (row0 >> 4) : row0, bar);
        ++iss_box;
        ++issued;
    };
    if constexpr (!MOE) {
        // weights never come from the preceding kernel: request them before the dependency
        // wait; x may, so only an L2 prefetch of this CTA's K range of it goes out before it
        iss_left = ie - ib;
        iw = first;
        if (tid == 0) trace_word(p.trace_slot, 33, static_cast<unsigned long long>(clock64()));
        if (lane == 0)
            for (int s = 0; s < min(stages, NVFP4_DENSE_EARLY); ++s) {
                issue_next();
                if (tid == 0 && s == 0) trace_word(p.trace_slot, 34, static_cast<unsigned long long>(clock64()));
            }
        if (tid == 0) trace_word(p.trace_slot, 35, static_cast<unsigned long long>(clock64()));
        if constexpr (SD) {
            // the table is a weight too: built before the dependency wait
            build_pair_table(reinterpret_cast<uint32_t*>(sbase + p.sdtab_off), p.sd_dict, tid, tk::kThreads);
            __syncthreads();
        }
        if (warp == tk::kWarps - 1 && lane < p.M) {
            const int kb = c_lo * NC * 256, kbytes = c_n * NC * 512;
            const uint16_t* xr = p.x + static_cast<int64_t>(lane) * p.K + kb;
            prefetch_l2_bulk(xr, static_cast<uint32_t>(kbytes));
            prefetch_l2(xr);  // through this SM's own path too, so its address translation is warm
        }
    } else {
        // which experts and rows are needed is known only from the ids: prefetch them and x
        if (warp == tk::kWarps - 1 && lane == 0) prefetch_l2(p.ids);
        const int xrows_all = p.x_per_slot ? p.slots : (p.slots + p.top_k - 1) / p.top_k;
        if (warp == tk::kWarps - 2 && lane < xrows_all) {
            const int kb = c_lo * NC * 256, kbytes = c_n * NC * 512;
            prefetch_l2_bulk(p.x + static_cast<int64_t>(lane) * p.K + kb, static_cast<uint32_t>(kbytes));
        }
    }
    if (tid == 0) trace_phase(p.trace_slot, 1);
    pdl_launch_dependents();
#if NVFP4_PHASE_TRACE && NVFP4_TRACE_BOX_LANDED
    // when the first box, requested before the dependency wait, lands (thread 0 waits for it
    // here, so this build delays warp 0 until then)
    if constexpr (!MOE)
        if (tid == 0 && ib < ie && nb > 0 && mbar_wait(&bars[0], 0, p.wait_ns))
            trace_word(p.trace_slot, 36, global_ns());
#endif
    pdl_wait();
    if (tid == 0) trace_phase(p.trace_slot, 2);

    int M = p.M;                 // x rows staged by this CTA
    const int* rowsel = nullptr; // their global row numbers (MoE)
    if constexpr (MOE) {
        // the expert ids may come from the preceding kernel: groups, items and weights only now
        if (warp == 0) tile_moe_groups(p, tab, lane);
        __syncthreads();
        unit_range(tab->n_groups * p.ipg);
        set_first();
        if (warp == 0 && ib < ie) tile_moe_rows(p, tab, ib / p.ipg, (ie - 1) / p.ipg, lane);
        iss_left = ie - ib;
        iw = first;
        __syncthreads();
        M = ib < ie ? tab->nrows : 0;
        rowsel = tab->rows;
        if (tid == 0) trace_word(p.trace_slot, 36, static_cast<unsigned long long>(clock64()));
    }

    // x for this warp's K slice, staged by the tpi warps that share the slice
    const uint32_t slice_bytes = static_cast<uint32_t>(p.M) * p.sstride;  // p.M: staged-row capacity
    uint8_t* const xs = sbase + p.x_off + kslice * slice_bytes;
    float* const e2 = reinterpret_cast<float*>(sbase + p.misc_off) + kslice * 8;
    // per slice: 16 words of extremes for the scaled staging, then 8 words of votes
    uint32_t* const gmax = reinterpret_cast<uint32_t*>(sbase + p.misc_off + tk::kWarps * 32) + kslice * 32;
    const int k0 = b_lo * NC * 256, kn = nb * NC * 256;
    const int xbar = p.tpi > 1 ? 2 + kslice : -1;
    bool lossy = false;
    float e2v = 1.f;
    bool staged = M == 0;
    if (M > 0) {
        if (NVFP4_STAGE_BULK)
            staged = stage_x_bulk(p.x, rowsel, M, p.K, k0, kn, xs, p.sstride, gmax + 16,
                                  reinterpret_cast<uint64_t*>(gmax + 24), tin, p.tpi, xbar, lane, p.wait_ns);
        else
            staged = stage_x_direct(p.x, rowsel, M, p.K, k0, kn, xs, p.sstride, gmax + 16, tin, p.tpi, xbar, lane,
                                    [] {});
    }
    if (!staged) {
        lossy = stage_x_slice(p.x, rowsel, M, p.K, k0, kn, xs, p.sstride, e2, gmax, tin, p.tpi, xbar, lane);
        e2v = e2[0];
    }
    if (tid == 0) trace_phase(p.trace_slot, 3);
    if constexpr (MOE) {
        // the weights of this CTA's experts: issued after staging, because a thread that issues
        // bulk copies can stall while the copy engine is busy, and staging waits for every warp
        if (lane == 0)
            for (int s = 0; s < stages; ++s) issue_next();
    } else {
        if (lane == 0)  // the rest of the ring, when only part of it went out before the wait
            for (int s = min(stages, NVFP4_DENSE_EARLY); s < stages; ++s) issue_next();
    }
    if (tid == 0) trace_word(p.trace_slot, 37, static_cast<unsigned long long>(clock64()));
    const bool use_f32 = lossy || p.force_f32;
    if (use_f32 && M > 0 && tin == 0 && lane == 0) atomicAdd(&g_fp32_fallbacks, 1ull);
    bool traced_first = false;

    const int g = lane >> 2;
    const int ra = tile_row_perm<NC>(g), rb = ra + 8;
    const uint32_t xslice = base + p.x_off + kslice * slice_bytes;
    uint32_t xa = xslice + static_cast<uint32_t>(min(g, max(M - 1, 0))) * p.sstride;
    const int m0 = 2 * t;
    const float e2s = use_f32 ? 1.f : e2v;  // the slice's power of two
    float* const red = reinterpret_cast<float*>(sbase + p.red_off);
    const uint64_t budget = p.wait_ns;
    bool dead = false;

    TileItemWalk cw = first;
    for (int item = ib; item < ie; ++item, cw.next(p.ipg)) {
        const int grp = cw.grp;
        const int tile = cw.t * p.tpi + tin;
        const bool valid = tile < p.tiles;
        int ncols = p.M;                       // output columns of this item
        const int* xrow = nullptr;             // global x row of each column (fp32 path)
        if constexpr (MOE) {
            ncols = tab->count[grp];
            xrow = tab->xrow[grp];
            xa = xslice + static_cast<uint32_t>(tab->col[grp][min(g, ncols - 1)]) * p.sstride;
        }
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        if (valid && !dead) {
            float dd[kTileChains][4];
#pragma unroll
            for (int c = 0; c < kTileChains; ++c)
#pragma unroll
                for (int i = 0; i < 4; ++i) dd[c][i] = 0.f;
            float acc[16];
            if (use_f32) {
#pragma unroll
                for (int i = 0; i < 16; ++i) acc[i] = 0.f;
            }
            for (int b = 0; b < nb; ++b) {
                const uint32_t st = cons_st;
                const uint32_t ph = cons_ph;
                if (NVFP4_PHASE_TRACE && !MOE && tid == 0 && !traced_first)
                    trace_word(p.trace_slot, 38, static_cast<unsigned long long>(clock64()));
                // a zero budget takes the timeout path deterministically (copies issued before
                // x staging have usually landed by now, so one poll would succeed)
                if (!__all_sync(0xffffffffu, budget != 0 && mbar_wait(&bars[st], ph, budget))) {
                    dead = true;  // warp-uniform: stop computing, keep the CTA's barrier count
                    break;
                }
                if (NVFP4_PHASE_TRACE && !MOE && tid == 0 && !traced_first)
                    trace_word(p.trace_slot, 39, static_cast<unsigned long long>(clock64()));
                if (NVFP4_PHASE_TRACE && lane == 0 && !traced_first) {
                    if (warp == 0) trace_phase(p.trace_slot, 4);
                    else trace_word(p.trace_slot, 24 + warp, global_ns());
                    traced_first = true;
                }
                if (!use_f32) {
                    tile_slot_mma<NC, SD>(ring_w + st * kWBox, ring_s + st * kSBox, xa, b * NC * 2, ra, t, dd,
                                          base + p.sdtab_off);
                } else {
                    tile_slot_f32<NC, SD>(ring_w + st * kWBox, ring_s + st * kSBox, p.x, xrow, p.K, ncols,
                                          (b_lo + b) * NC, ra, t, acc, base + p.sdtab_off);
                }
                cons_advance();
                __syncwarp();
                if (lane == 0) issue_next();
            }
            if (use_f32) {
#pragma unroll
                for (int i = 0; i < 16; ++i) {
                    acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 1);
                    acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 2);
                }
                // the MMA's accumulator layout: (ra, 2t), (ra, 2t+1), (rb, 2t), (rb, 2t+1)
#pragma unroll
                for (int m = 0; m < 8; ++m) {
                    if (m == m0) { d[0] = acc[m]; d[2] = acc[8 + m]; }
                    if (m == m0 + 1) { d[1] = acc[m]; d[3] = acc[8 + m]; }
                }
            } else {
#pragma unroll
                for (int c = 0; c < kTileChains; ++c)
#pragma unroll
                    for (int i = 0; i < 4; ++i) d[i] += dd[c][i];
            }
            if (dead) raise_status(NVFP4_DEV_TIMEOUT, nullptr);
        }
        // this slice's partial sums in x units: times its power of two
#pragma unroll
        for (int i = 0; i < 4; ++i) d[i] *= e2s;
        float gs;
        if constexpr (MOE) gs = __ldg(p.g_dev + tab->expert[grp]);
        else gs = p.g[grp];
        // where output (column m, row `row` of the group) goes
        auto out_at = [&](int m, int row) -> int64_t {
            if constexpr (MOE) return static_cast<int64_t>(tab->slot[grp][m]) * p.N + row;
            else return m * p.ldy + static_cast<int64_t>(grp) * p.N + row;
        };
        const int par = (item - ib) & 1;
        float* const cpart = reinterpret_cast<float*>(sbase + p.cpart_off) + par * (tk::kWarps * 16 * 8);
        if constexpr (SWI) {
            // gate tile 2j and up tile 2j + 1 of this item meet in cpart ([tile * 16 + row][m]:
            // this CTA's sums over its K range), then every output combines its pair
            const int outs = p.tpi * 16 * ncols;
            const int pair_outs = (p.tpi >> 1) * 16 * ncols;
            if (ksplit == 1) {
                float* cp = cpart + tin * 128;
                cp[ra * 8 + m0] = d[0];
                cp[ra * 8 + m0 + 1] = d[1];
                cp[rb * 8 + m0] = d[2];
                cp[rb * 8 + m0 + 1] = d[3];
            } else {
                float* rbuf = red + par * tk::kRedFloats + warp * 128;
                rbuf[ra * 8 + m0] = d[0];
                rbuf[ra * 8 + m0 + 1] = d[1];
                rbuf[rb * 8 + m0] = d[2];
                rbuf[rb * 8 + m0 + 1] = d[3];
                named_bar_sync(1, tk::kThreads);
                const float* rb0 = red + par * tk::kRedFloats;
                for (int i = tid; i < outs; i += tk::kThreads) {
                    const int ti = i / (16 * ncols), rem = i - ti * 16 * ncols;
                    const int r = rem / ncols, m = rem - r * ncols;
                    float sum = 0.f;
                    for (int j = 0; j < ksplit; ++j) sum += rb0[((ti << p.ksplit_log2) + j) * 128 + r * 8 + m];
                    cpart[ti * 128 + r * 8 + m] = sum;
                }
            }
            int o_lo = 0, o_hi = pair_outs, o_step = tk::kThreads;
            if (S == 1) {
                named_bar_sync(1, tk::kThreads);
            } else {
                // the cluster's K ranges: rank r combines the r-th share of the outputs, adding
                // the ranks' sums in rank order (DSMEM)
                cluster_sync_all();
                o_lo = (rank * pair_outs) >> p.s_log2;
                o_hi = ((rank + 1) * pair_outs) >> p.s_log2;
            }
            for (int i = o_lo + tid; i < o_hi; i += o_step) {
                const int pi = i / (16 * ncols), rem = i - pi * 16 * ncols;
                const int r = rem / ncols, m = rem - r * ncols;
                const int jt = cw.t * (p.tpi >> 1) + pi, row = jt * 16 + r;  // output tile, row
                if (2 * jt < p.tiles && row < p.N) {
                    const float* cg = cpart + (2 * pi) * 128 + r * 8 + m;
                    float sg = 0.f, su = 0.f;
                    if (S == 1) {
                        sg = cg[0];
                        su = cg[128];
                    } else {
                        for (int j = 0; j < S; ++j) {
                            sg += ld_cluster_f32(cg, j);
                            su += ld_cluster_f32(cg + 128, j);
                        }
                    }
                    store_out(p.y, m * p.ldy + row, swiglu_f32(sg * p.g[0], su * p.g[1], p.clamp), p.out_bf16);
                }
            }
            continue;
        }
        if (ksplit == 1 && S == 1) {
            if (valid) {
                const int rowa = tile * 16 + ra, rowb = tile * 16 + rb;
                if (m0 < ncols) {
                    if (rowa < p.N) store_out(p.y, out_at(m0, rowa), d[0] * gs, p.out_bf16);
                    if (rowb < p.N) store_out(p.y, out_at(m0, rowb), d[2] * gs, p.out_bf16);
                }
                if (m0 + 1 < ncols) {
                    if (rowa < p.N) store_out(p.y, out_at(m0 + 1, rowa), d[1] * gs, p.out_bf16);
                    if (rowb < p.N) store_out(p.y, out_at(m0 + 1, rowb), d[3] * gs, p.out_bf16);
                }
            }
            continue;
        }
        const int outs = p.tpi * 16 * ncols;  // this item's outputs, as (tile, row, m)
        if (ksplit == 1) {
            // one warp per tile: its sums are this CTA's part (cpart is [tile * 16 + row][m])
            float* cp = cpart + tin * 128;
            cp[ra * 8 + m0] = d[0];
            cp[ra * 8 + m0 + 1] = d[1];
            cp[rb * 8 + m0] = d[2];
            cp[rb * 8 + m0 + 1] = d[3];
        } else {
            float* rbuf = red + par * tk::kRedFloats + warp * 128;
            rbuf[ra * 8 + m0] = d[0];
            rbuf[ra * 8 + m0 + 1] = d[1];
            rbuf[rb * 8 + m0] = d[2];
            rbuf[rb * 8 + m0 + 1] = d[3];
            named_bar_sync(1, tk::kThreads);
            const float* rb0 = red + par * tk::kRedFloats;
            for (int i = tid; i < outs; i += tk::kThreads) {
                const int ti = i / (16 * ncols), rem = i - ti * 16 * ncols;
                const int r = rem / ncols, m = rem - r * ncols;
                float sum = 0.f;
                for (int j = 0; j < ksplit; ++j) sum += rb0[((ti << p.ksplit_log2) + j) * 128 + r * 8 + m];
                if (S == 1) {
                    const int tl = cw.t * p.tpi + ti, row = tl * 16 + r;
                    if (tl < p.tiles && row < p.N) store_out(p.y, out_at(m, row), sum * gs, p.out_bf16);
                } else {
                    cpart[ti * 128 + r * 8 + m] = sum;
                }
            }
            if (S == 1) continue;
        }
        // the cluster's K ranges: after the barrier, rank r adds the r-th share of the outputs
        // over all ranks in rank order (DSMEM), so the sum does not depend on timing
        cluster_sync_all();
        const int o_lo = (rank * outs) >> p.s_log2, o_hi = ((rank + 1) * outs) >> p.s_log2;
        for (int i = o_lo + tid; i < o_hi; i += tk::kThreads) {
            const int ti = i / (16 * ncols), rem = i - ti * 16 * ncols;
            const int r = rem / ncols, m = rem - r * ncols;
            const int tl = cw.t * p.tpi + ti, row = tl * 16 + r;
            if (tl < p.tiles && row < p.N) {
                float sum = 0.f;
                for (int j = 0; j < S; ++j) sum += ld_cluster_f32(cpart + ti * 128 + r * 8 + m, j);
                store_out(p.y, out_at(m, row), sum * gs, p.out_bf16);
            }
        }
    }
    if (lane == 0) trace_word(p.trace_slot, 16 + warp, global_ns());
    if (tid == 0) trace_phase(p.trace_slot, 6);
    // no CTA may leave while another rank of its cluster can still read its partial sums
    if (S > 1) cluster_sync_all();
    // copies still in flight (only after a timeout) must land before the CTA exits
    if (lane == 0) {
        while (consumed < issued) {
            mbar_wait(&bars[cons_st], cons_ph, kDrainWaitNs);
            cons_advance();
        }
    }
    __syncwarp();
    if (tid == 0) trace_phase(p.trace_slot, 7);
    trace_flush(p.trace_slot, tid);
}

// ------------------------------------------------------------------ the FFN block in one launch

// The shared-expert FFN group of "glm-5.3-flash-nvfp4-tp3-512k--gb10 graph.json" (block l3.moe:
// shared_gate_up, shared_clamp, shared_act, shared_down) as one launch. Phase A is the gate/up
// GEMV with the fused SwiGLU (wmap/smap [0] gate, [1] up; y = h, bf16 [M, I]); phase B is the
// down GEMV (wmap/smap [0]; x = h; y = the block's output). Both phases use one ring (NC,
// stages), one grid with every CTA resident at once (two per SM) and no clusters.
//
// The phases meet through readiness counters instead of a grid barrier: phase B's warp with K
// slice s needs only h[:, slice s], which a known number of phase-A items write. Every A item,
// once its h rows are stored, adds one to its slice's counter (release); a B warp waits
// (acquire, bounded) until its slice's counter holds all of them. A items are dealt round-robin
// over the CTAs, so the low slices fill early, and B items go first to the CTAs with fewer A
// items. `sync` is the caller's workspace: word 0 counts the CTAs that are done with the
// counters, word 32 (s + 1) is slice s's counter (each in its own 128-byte line); the last CTA
// done sets them all back to zero for the next launch.
//
// A ninth warp does every release and acquire-release operation on these words, so no compute
// warp ever waits for a GPU-scope fence. After storing an item's h rows each compute warp adds
// one to a shared-memory count (release, CTA scope); the ninth warp waits (acquire) until all
// eight have, then counts the item in. Once all compute warps have passed their slice waits
// (a second shared count), it counts the CTA as done. Both shared counts only grow, so the
// ninth warp may fall any number of items behind.
struct FfnParams {
    TileParams a, b;
    uint32_t* sync;
};

constexpr int kFfnSyncBytes = 2048;   // workspace bytes before h: the counters' lines
constexpr int kFfnSlices = 8;         // B's K slices (one counter each)
constexpr int kFfnThreads = tk::kThreads + 32;  // 8 compute warps and the signalling warp
constexpr int64_t kFfnFusedMaxBytes = 12ll << 20;  // weights of the largest block run as one launch

#ifndef NVFP4_FFN_H_PRE
#define NVFP4_FFN_H_PRE 6  // loads in flight per lane when phase B stages h (one batch at M = 1, I = 12288)
#endif

// One phase's share of a warp: its tile within an item, its box range (K slice), and its CTA's
// items first, first + stride, ... (count of them). Phase A deals items round-robin (item i to
// CTA i mod units); phase B in reverse (item j to CTA units - 1 - j mod units), so B's items
// land first on the CTAs that drew one A item fewer.
struct FfnGeo {
    int tin, kslice, b_lo, nb, first, count, stride;
};

__host__ __device__ __forceinline__ FfnGeo ffn_geo(const TileParams& q, int warp, int unit, int units, bool rev) {
    FfnGeo g;
    const int ksplit = 1 << q.ksplit_log2;
    g.kslice = warp & (ksplit - 1);
    g.tin = warp >> q.ksplit_log2;
    g.b_lo = (g.kslice * q.nbox) >> q.ksplit_log2;
    g.nb = (((g.kslice + 1) * q.nbox) >> q.ksplit_log2) - g.b_lo;
    const int items = q.items_q * units + q.items_r;
    g.first = rev ? units - 1 - unit : unit;
    g.count = g.first < items ? (items - g.first + units - 1) / units : 0;
    g.stride = units;
    return g;
}

// Rows of h one phase-A item writes (its gate/up tile pairs x 16), and the A items whose rows
// fall in phase B's K slice s (slices start at multiples of 256 rows, which R divides).
__host__ __device__ __forceinline__ int ffn_item_rows(const TileParams& a) { return (a.tpi >> 1) * 16; }

__host__ __device__ __forceinline__ int ffn_slice_lo(const TileParams& b, int s, int nc) {
    return ((s * b.nbox) >> b.ksplit_log2) * nc * 256;
}

__host__ __device__ __forceinline__ int ffn_slice_items(const TileParams& a, const TileParams& b, int s, int nc) {
    const int lo = ffn_slice_lo(b, s, nc), hi = min(ffn_slice_lo(b, s + 1, nc), b.K);
    const int r = ffn_item_rows(a);
    return (hi - lo + r - 1) / r;
}

// B's K slice holding h row `row` (the slice whose range contains it).
__host__ __device__ __forceinline__ int ffn_slice_of(const TileParams& b, int row, int nc) {
    const int ks = 1 << b.ksplit_log2;
    int s = 0;
    while (s + 1 < ks && ffn_slice_lo(b, s + 1, nc) <= row) ++s;
    return s;
}

__device__ __forceinline__ uint32_t ld_acquire_gpu(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ uint32_t atom_add_acq_rel_gpu(uint32_t* p, uint32_t v) {
    uint32_t old;
    asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
    return old;
}

__device__ __forceinline__ void red_add_release_gpu(uint32_t* p, uint32_t v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void st_relaxed_gpu(uint32_t* p, uint32_t v) {
    asm volatile("st.relaxed.gpu.global.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

__device__ __forceinline__ void red_add_release_cta_shared(uint32_t* p, uint32_t v) {
    asm volatile("red.release.cta.shared::cta.add.u32 [%0], %1;" ::"r"(smem_addr(p)), "r"(v) : "memory");
}

__device__ __forceinline__ uint32_t ld_acquire_cta_shared(const uint32_t* p) {
    uint32_t v;
    asm volatile("ld.acquire.cta.shared::cta.u32 %0, [%1];" : "=r"(v) : "r"(smem_addr(p)) : "memory");
    return v;
}

// One thread waits (acquire, CTA scope) until the shared count *c reaches want, for at most
// `budget` ns. False when it ran out (the count is the CTA's own: only a defect leaves it short).
__device__ bool ffn_wait_shared(const uint32_t* c, uint32_t want, uint64_t budget) {
    if (ld_acquire_cta_shared(c) >= want) return true;
    const uint64_t t0 = global_ns();
    while (ld_acquire_cta_shared(c) < want) {
        if (global_ns() - t0 > budget) return false;
        __nanosleep(64);
    }
    return true;
}

// Waits (every lane, acquire) until *cnt >= want, for at most `budget` ns (0: one look).
// Returns whether it got there (uniform over the warp: all lanes read the same word, and the
// warp votes).
__device__ bool ffn_wait_count(const uint32_t* cnt, uint32_t want, uint64_t budget) {
    bool ok = ld_acquire_gpu(cnt) >= want;
    if (__all_sync(0xffffffffu, ok)) return true;
    const uint64_t t0 = global_ns();
    uint32_t ns = 32;
    for (;;) {
        ok = ld_acquire_gpu(cnt) >= want;
        if (__all_sync(0xffffffffu, ok)) return true;
        if (budget == 0 || global_ns() - t0 > budget) return false;
        __nanosleep(ns);
        ns = ns < 256 ? 2 * ns : 256;
    }
}

template <int NC>
__global__ void __launch_bounds__(kFfnThreads, 2) gemv_ffn_kernel(const __grid_constant__ FfnParams p) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t s_sig[2];  // compute warps that stored an A item's h rows / passed their slice wait
    constexpr uint32_t kWBox = NC * 2048;
    constexpr uint32_t kSBox = scale_box_bytes<NC, false>();
    const TileParams& A = p.a;
    const TileParams& B = p.b;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t = lane & 3;
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* const sbase = smem_raw + (base - raw_base);
    const int stages = A.stages;  // one ring for both phases
    uint64_t* const bars = reinterpret_cast<uint64_t*>(sbase + A.bar_off) + warp * tk::kMaxStages;
    const uint32_t ring_w = base + A.ring_w + static_cast<uint32_t>(warp * stages) * kWBox;
    const uint32_t ring_s = base + A.ring_s + static_cast<uint32_t>(warp * stages) * kSBox;
    const int slot = A.trace_slot;
    if (tid == 0) s_sig[0] = s_sig[1] = 0u;
    __syncthreads();
    trace_begin(tid);
    if (tid == 0) trace_phase(slot, 0);
    const int unit = blockIdx.x, units = gridDim.x;
    if (warp == tk::kWarps) {
        // the signalling warp: counts every A item into its B slice once the compute warps have
        // stored its h rows, then counts the CTA as done once they are past their slice waits
        pdl_launch_dependents();
        pdl_wait();
        const FfnGeo ga = ffn_geo(A, 0, unit, units, false);
        for (int j = 0; j < ga.count && lane == 0; ++j) {
            if (!ffn_wait_shared(&s_sig[0], static_cast<uint32_t>(tk::kWarps * (j + 1)), kDrainWaitNs))
                raise_status(NVFP4_DEV_INTERNAL, nullptr);
            const int item = ga.first + j * ga.stride;
            if (2 * item * (A.tpi >> 1) < A.tiles)
                red_add_release_gpu(p.sync + 32 * (1 + ffn_slice_of(B, item * ffn_item_rows(A), NC)), 1u);
        }
        if (lane == 0) {
            if (!ffn_wait_shared(&s_sig[1], static_cast<uint32_t>(tk::kWarps), kDrainWaitNs))
                raise_status(NVFP4_DEV_INTERNAL, nullptr);
            // the last CTA done puts the counters back to zero: every CTA counted its A items and
            // passed its waits before it counts itself here (acq_rel chain on word 0)
            const uint32_t done = atom_add_acq_rel_gpu(p.sync, 1u);
            if (done == static_cast<uint32_t>(units) - 1u) {
                for (int s = 0; s < kFfnSlices; ++s) st_relaxed_gpu(p.sync + 32 * (1 + s), 0u);
                st_relaxed_gpu(p.sync, 0u);
            }
        }
        __syncwarp();
        trace_flush(slot, tid);
        return;
    }
    if (NVFP4_PREFETCH_TMAP && warp == 0 && lane < 3) prefetch_tmap(lane < 2 ? &A.wmap[lane] : &B.wmap[0]);
    if (NVFP4_PREFETCH_TMAP && warp == 1 && lane < 3) prefetch_tmap(lane < 2 ? &A.smap[lane] : &B.smap[0]);
    const FfnGeo ga = ffn_geo(A, warp, unit, units, false);
    const FfnGeo gb = ffn_geo(B, warp, unit, units, true);
    if (lane == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncwarp();

    // lane 0's issue cursor walks phase A's boxes, then phase B's: neither depends on x or h, so
    // B's first boxes stream in while A finishes
    int iph = 0;
    int iss_j = 0, iss_box = 0;
    uint32_t issued = 0, consumed = 0;
    uint32_t iss_st = 0, cons_st = 0, cons_ph = 0;
    auto cons_advance = [&]() {
        ++consumed;
        if (++cons_st == static_cast<uint32_t>(stages)) {
            cons_st = 0;
            cons_ph ^= 1u;
        }
    };
    auto issue_next = [&]() {
        for (;;) {
            if (iph == 2) return;
            const bool pa = iph == 0;
            const FfnGeo& g = pa ? ga : gb;
            const int tpi = pa ? A.tpi : B.tpi, tiles = pa ? A.tiles : B.tiles;
            while (iss_j < g.count && (iss_box >= g.nb || (g.first + iss_j * g.stride) * tpi + g.tin >= tiles)) {
                ++iss_j;
                iss_box = 0;
            }
            if (iss_j < g.count) break;
            iph = pa ? 1 : 2;
            iss_j = 0;
            iss_box = 0;
        }
        const uint32_t st = iss_st;
        if (++iss_st == static_cast<uint32_t>(stages)) iss_st = 0;
        const uint32_t bar = smem_addr(&bars[st]);
        mbar_arrive_expect_tx(&bars[st], kWBox + scale_box_tx<NC, false>());
        if (iph == 0) {
            const int tile = (ga.first + iss_j * ga.stride) * A.tpi + ga.tin;  // tiles alternate gate, up
            const int seg = (ga.b_lo + iss_box) * NC, row0 = (tile >> 1) * 16;
            tma_load_3d(ring_w + st * kWBox, &A.wmap[tile & 1], 0, seg, row0, bar);
            tma_load_3d(ring_s + st * kSBox, &A.smap[tile & 1], 0, seg, row0, bar);
        } else {
            const int tile = (gb.first + iss_j * gb.stride) * B.tpi + gb.tin;
            const int seg = (gb.b_lo + iss_box) * NC;
            tma_load_3d(ring_w + st * kWBox, &B.wmap[0], 0, seg, tile * 16, bar);
            tma_load_3d(ring_s + st * kSBox, &B.smap[0], 0, seg, tile * 16, bar);
        }
        ++iss_box;
        ++issued;
    };
    // gate/up weights before the dependency wait (x may come from the preceding kernel; only an
    // L2 prefetch of it goes out before the wait)
    if (lane == 0)
        for (int s = 0; s < min(stages, NVFP4_DENSE_EARLY); ++s) issue_next();
    const int M = A.M;
    if (warp == tk::kWarps - 1 && lane < M) {
        const uint16_t* xr = A.x + static_cast<int64_t>(lane) * A.K;
        prefetch_l2_bulk(xr, static_cast<uint32_t>(A.K) * 2u);
        prefetch_l2(xr);
    }
    if (tid == 0) trace_phase(slot, 1);
    pdl_launch_dependents();
    pdl_wait();
    if (tid == 0) trace_phase(slot, 2);

    bool dead = false;  // warp-uniform: a wait ran out of time
    // One phase: stage this warp's K slice of x (A) or h (B), then run the CTA's items.
    auto phase = [&](auto swi_tag, const TileParams& q, const FfnGeo& g) {
        constexpr bool SWI = decltype(swi_tag)::value;
        const int ksplit = 1 << q.ksplit_log2;
        const int kslice = g.kslice, tin = g.tin;
        const uint32_t slice_bytes = static_cast<uint32_t>(M) * q.sstride;
        uint8_t* const xs = sbase + q.x_off + kslice * slice_bytes;
        float* const e2 = reinterpret_cast<float*>(sbase + q.misc_off) + kslice * 8;
        uint32_t* const gmax = reinterpret_cast<uint32_t*>(sbase + q.misc_off + tk::kWarps * 32) + kslice * 32;
        const int k0 = g.b_lo * NC * 256, kn = g.nb * NC * 256;
        const int xbar = q.tpi > 1 ? 2 + kslice : -1;
        if constexpr (!SWI) {
            // h[:, slice] is complete once every A item of the slice has counted itself in; the
            // staging runs even after a timeout, so the slice's warps keep their barrier counts
            if (g.count > 0 && !dead &&
                !ffn_wait_count(p.sync + 32 * (1 + kslice), static_cast<uint32_t>(ffn_slice_items(A, B, kslice, NC)),
                                q.wait_ns)) {
                dead = true;
                if (lane == 0) raise_status(NVFP4_DEV_TIMEOUT, nullptr);
            }
            if (tid == 0) trace_word(slot, 38, global_ns());
            __syncwarp();  // every lane is done reading the counters
            if (lane == 0) red_add_release_cta_shared(&s_sig[1], 1u);
        }
        bool lossy = false;
        float e2v = 1.f;
        // h was written by other CTAs of this launch: read it through L2 only
        const bool staged = SWI ? stage_x_direct<NVFP4_STAGE_PRE, false>(q.x, nullptr, M, q.K, k0, kn, xs, q.sstride,
                                                                         gmax + 16, tin, q.tpi, xbar, lane, [] {})
                                : stage_x_direct<NVFP4_FFN_H_PRE, true>(q.x, nullptr, M, q.K, k0, kn, xs, q.sstride,
                                                                        gmax + 16, tin, q.tpi, xbar, lane, [] {});
        if (!staged) {
            lossy = SWI ? stage_x_slice<false>(q.x, nullptr, M, q.K, k0, kn, xs, q.sstride, e2, gmax, tin, q.tpi,
                                               xbar, lane)
                        : stage_x_slice<true>(q.x, nullptr, M, q.K, k0, kn, xs, q.sstride, e2, gmax, tin, q.tpi,
                                              xbar, lane);
            e2v = e2[0];
        }
        if constexpr (SWI) {
            if (tid == 0) trace_phase(slot, 3);
            if (lane == 0)  // the rest of the ring
                for (int s = min(stages, NVFP4_DENSE_EARLY); s < stages; ++s) issue_next();
        } else {
            if (tid == 0) trace_word(slot, 39, global_ns());
        }
        const bool use_f32 = lossy || q.force_f32;
        if (use_f32 && tin == 0 && lane == 0) atomicAdd(&g_fp32_fallbacks, 1ull);
        const int g8 = lane >> 2;
        const int ra = tile_row_perm<NC>(g8), rb = ra + 8;
        const uint32_t xa = base + q.x_off + kslice * slice_bytes + static_cast<uint32_t>(min(g8, M - 1)) * q.sstride;
        const int m0 = 2 * t;
        const float e2s = use_f32 ? 1.f : e2v;
        float* const red = reinterpret_cast<float*>(sbase + q.red_off);
        const uint64_t budget = q.wait_ns;
        bool traced_first = false;
        for (int j = 0; j < g.count; ++j) {
            const int item = g.first + j * g.stride;
            const int tile = item * q.tpi + tin;
            const bool valid = tile < q.tiles;
            float d[4] = {0.f, 0.f, 0.f, 0.f};
            if (valid && !dead) {
                float dd[kTileChains][4];
#pragma unroll
                for (int c = 0; c < kTileChains; ++c)
#pragma unroll
                    for (int i = 0; i < 4; ++i) dd[c][i] = 0.f;
                float acc[16];
                if (use_f32) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
                }
                for (int b = 0; b < g.nb; ++b) {
                    const uint32_t st = cons_st;
                    const uint32_t ph = cons_ph;
                    if (!__all_sync(0xffffffffu, budget != 0 && mbar_wait(&bars[st], ph, budget))) {
                        dead = true;  // stop computing, keep the CTA's barrier counts
                        break;
                    }
                    if (NVFP4_PHASE_TRACE && SWI && warp == 0 && lane == 0 && !traced_first) {
                        trace_phase(slot, 4);
                        traced_first = true;
                    }
                    if (!use_f32) {
                        tile_slot_mma<NC>(ring_w + st * kWBox, ring_s + st * kSBox, xa, b * NC * 2, ra, t, dd);
                    } else {
                        tile_slot_f32<NC, false, !SWI>(ring_w + st * kWBox, ring_s + st * kSBox, q.x, nullptr, q.K,
                                                       M, (g.b_lo + b) * NC, ra, t, acc);
                    }
                    cons_advance();
                    __syncwarp();
                    if (lane == 0) issue_next();
                }
                if (use_f32) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 1);
                        acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 2);
                    }
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        if (m == m0) { d[0] = acc[m]; d[2] = acc[8 + m]; }
                        if (m == m0 + 1) { d[1] = acc[m]; d[3] = acc[8 + m]; }
                    }
                } else {
#pragma unroll
                    for (int c = 0; c < kTileChains; ++c)
#pragma unroll
                        for (int i = 0; i < 4; ++i) d[i] += dd[c][i];
                }
                if (dead && lane == 0) raise_status(NVFP4_DEV_TIMEOUT, nullptr);
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) d[i] *= e2s;
            const int par = j & 1;
            float* const cpart = reinterpret_cast<float*>(sbase + q.cpart_off) + par * (tk::kWarps * 16 * 8);
            if constexpr (SWI) {
                // gate tile 2j and up tile 2j + 1 meet in cpart ([tile * 16 + row][m]), then every
                // output combines its pair into one bf16 h
                const int outs = q.tpi * 16 * M;
                const int pair_outs = (q.tpi >> 1) * 16 * M;
                if (ksplit == 1) {
                    float* cp = cpart + tin * 128;
                    cp[ra * 8 + m0] = d[0];
                    cp[ra * 8 + m0 + 1] = d[1];
                    cp[rb * 8 + m0] = d[2];
                    cp[rb * 8 + m0 + 1] = d[3];
                } else {
                    float* rbuf = red + par * tk::kRedFloats + warp * 128;
                    rbuf[ra * 8 + m0] = d[0];
                    rbuf[ra * 8 + m0 + 1] = d[1];
                    rbuf[rb * 8 + m0] = d[2];
                    rbuf[rb * 8 + m0 + 1] = d[3];
                    named_bar_sync(1, tk::kThreads);
                    const float* rb0 = red + par * tk::kRedFloats;
                    for (int i = tid; i < outs; i += tk::kThreads) {
                        const int ti = i / (16 * M), rem = i - ti * 16 * M;
                        const int r = rem / M, m = rem - r * M;
                        float sum = 0.f;
                        for (int jj = 0; jj < ksplit; ++jj) sum += rb0[((ti << q.ksplit_log2) + jj) * 128 + r * 8 + m];
                        cpart[ti * 128 + r * 8 + m] = sum;
                    }
                }
                named_bar_sync(1, tk::kThreads);
                for (int i = tid; i < pair_outs; i += tk::kThreads) {
                    const int pi = i / (16 * M), rem = i - pi * 16 * M;
                    const int r = rem / M, m = rem - r * M;
                    const int jt = item * (q.tpi >> 1) + pi, row = jt * 16 + r;  // output tile, row
                    if (2 * jt < q.tiles && row < q.N) {
                        const float* cg = cpart + (2 * pi) * 128 + r * 8 + m;
                        store_out(q.y, m * q.ldy + row, swiglu_f32(cg[0] * q.g[0], cg[128] * q.g[1], q.clamp),
                                  q.out_bf16);
                    }
                }
                // the item's h rows are stored: the signalling warp counts them in once all eight
                // warps have said so (the warp barrier orders the lanes' stores before lane 0's
                // release)
                __syncwarp();
                if (lane == 0) red_add_release_cta_shared(&s_sig[0], 1u);
            } else {
                const float gs = q.g[0];
                if (ksplit == 1) {
                    if (valid) {
                        const int rowa = tile * 16 + ra, rowb = tile * 16 + rb;
                        if (m0 < M) {
                            if (rowa < q.N) store_out(q.y, m0 * q.ldy + rowa, d[0] * gs, q.out_bf16);
                            if (rowb < q.N) store_out(q.y, m0 * q.ldy + rowb, d[2] * gs, q.out_bf16);
                        }
                        if (m0 + 1 < M) {
                            if (rowa < q.N) store_out(q.y, (m0 + 1) * q.ldy + rowa, d[1] * gs, q.out_bf16);
                            if (rowb < q.N) store_out(q.y, (m0 + 1) * q.ldy + rowb, d[3] * gs, q.out_bf16);
                        }
                    }
                } else {
                    const int outs = q.tpi * 16 * M;
                    float* rbuf = red + par * tk::kRedFloats + warp * 128;
                    rbuf[ra * 8 + m0] = d[0];
                    rbuf[ra * 8 + m0 + 1] = d[1];
                    rbuf[rb * 8 + m0] = d[2];
                    rbuf[rb * 8 + m0 + 1] = d[3];
                    named_bar_sync(1, tk::kThreads);
                    const float* rb0 = red + par * tk::kRedFloats;
                    for (int i = tid; i < outs; i += tk::kThreads) {
                        const int ti = i / (16 * M), rem = i - ti * 16 * M;
                        const int r = rem / M, m = rem - r * M;
                        float sum = 0.f;
                        for (int jj = 0; jj < ksplit; ++jj) sum += rb0[((ti << q.ksplit_log2) + jj) * 128 + r * 8 + m];
                        const int tl = item * q.tpi + ti, row = tl * 16 + r;
                        if (tl < q.tiles && row < q.N) store_out(q.y, m * q.ldy + row, sum * gs, q.out_bf16);
                    }
                }
            }
        }
    };

    phase(std::integral_constant<bool, true>{}, A, ga);
    if (tid == 0) trace_phase(slot, 5);
    phase(std::integral_constant<bool, false>{}, B, gb);
    if (tid == 0) trace_phase(slot, 6);
    // copies still in flight (only after a timeout) land before the CTA exits
    if (lane == 0) {
        while (consumed < issued) {
            mbar_wait(&bars[cons_st], cons_ph, kDrainWaitNs);
            cons_advance();
        }
    }
    __syncwarp();
    if (tid == 0) trace_phase(slot, 7);
    trace_flush(slot, tid);
}

#ifndef NVFP4_MOE_EARLY
#define NVFP4_MOE_EARLY 1  // weight slots a MoE warp requests before x staging (the rest after it)
#endif
#ifndef NVFP4_SK_GROUP_ALIGNED
#define NVFP4_SK_GROUP_ALIGNED 1  // 1: the planner may keep each stream-K CTA inside one expert group (0: never)
#endif

// Stream-K form of the warp-tile kernel, for launches with many tiles per CTA (all 8 warps
// share one K range: the whole of K). The jobs (group, 16-row tile), group-major, are split
// into balanced contiguous ranges of whole jobs per CTA; inside a CTA the jobs' TMA boxes are
// split evenly over the 8 warps, so a warp's range may start or end inside a job. A warp that
// covers a whole job stores it directly. A job split between warps leaves a partial record (at
// most two per warp: its first and its last job; the first is held in registers) that the warp
// writes into its own ring once all its copies are consumed. After one CTA barrier the warp
// that holds a job's first box adds the records of the following warps in warp order and
// stores the sum. Balance is one TMA box per warp instead of one item per CTA.
template <int NC, bool MOE, bool SD = false>
__global__ void __launch_bounds__(tk::kThreads, 2) gemv_tile_sk_kernel(const __grid_constant__ TileParams p) {
    extern __shared__ uint8_t smem_raw[];
    constexpr uint32_t kWBox = NC * 2048;
    constexpr uint32_t kSBox = scale_box_bytes<NC, SD>();
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int t = lane & 3;
    const uint32_t raw_base = smem_addr(smem_raw);
    const uint32_t base = (raw_base + 1023u) & ~1023u;
    uint8_t* const sbase = smem_raw + (base - raw_base);
    const int stages = p.stages, nbox = p.nbox, tiles = p.tiles;
    uint64_t* const bars = reinterpret_cast<uint64_t*>(sbase + p.bar_off) + warp * tk::kMaxStages;
    const uint32_t ring_w = base + p.ring_w + static_cast<uint32_t>(warp * stages) * kWBox;
    const uint32_t ring_s = base + p.ring_s + static_cast<uint32_t>(warp * stages) * kSBox;
    TileMoe* const tab = reinterpret_cast<TileMoe*>(sbase + p.moe_off);
    trace_begin(tid);
    if (tid == 0) trace_phase(p.trace_slot, 0);
    if (NVFP4_PREFETCH_TMAP && warp == 0 && lane < 4) prefetch_tmap(lane < 2 ? &p.wmap[lane] : &p.smap[lane - 2]);
    // partial records of warp w: the first 1 KB of its own ring, free once its boxes are consumed
    auto rec_of = [&](int w, int slot) -> float* {
        return reinterpret_cast<float*>(sbase + p.ring_w + static_cast<uint32_t>(w * stages) * kWBox) + slot * 128;
    };

    if (lane == 0) {
        for (int s = 0; s < stages; ++s) mbar_init(&bars[s], 1);
        fence_barrier_init();
    }
    __syncwarp();

    // this CTA's jobs [j0, j1) and this warp's boxes [bs, be) of them (box b: job j0 + b / nbox)
    int j0 = 0, j1 = 0, bs = 0, be = 0;
    auto set_ranges = [&](int jobs) {
        const int q = jobs / static_cast<int>(gridDim.x), r = jobs - q * static_cast<int>(gridDim.x);
        j0 = blockIdx.x * q + min(static_cast<int>(blockIdx.x), r);
        j1 = j0 + q + (static_cast<int>(blockIdx.x) < r ? 1 : 0);
        const int total = (j1 - j0) * nbox;
        bs = (warp * total) >> 3;
        be = ((warp + 1) * total) >> 3;
    };
    // issue cursor (lane 0)
    int is_b = 0, is_box = 0, is_tile = 0, is_grp = 0;
    uint32_t issued = 0, consumed = 0;
    // ring positions kept incrementally (the ring depth is a launch parameter: no divisions)
    uint32_t iss_st = 0, cons_st = 0, cons_ph = 0;
    auto cons_advance = [&]() {
        ++consumed;
        if (++cons_st == static_cast<uint32_t>(stages)) {
            cons_st = 0;
            cons_ph ^= 1u;
        }
    };
    auto start_cursor = [&]() {
        is_b = bs;
        const int job = j0 + bs / nbox;
        is_box = bs - (bs / nbox) * nbox;
        is_grp = job / tiles;
        is_tile = job - is_grp * tiles;
    };
    int gw0 = 0;  // MoE: the group held by entry 0 of the tables
    auto issue_next = [&]() {
        if (is_b >= be) return;
        const uint32_t st = iss_st;
        if (++iss_st == static_cast<uint32_t>(stages)) iss_st = 0;
        const uint32_t bar = smem_addr(&bars[st]);
        mbar_arrive_expect_tx(&bars[st], kWBox + scale_box_tx<NC, SD>());
        int row0 = is_tile * 16, map = is_grp, srow = SD ? is_tile : row0;
        if constexpr (MOE) {
            row0 += tab->expert[is_grp - gw0] * p.N;
            srow += tab->expert[is_grp - gw0] * (SD ? p.sd_tiles : p.N);
            map = 0;
        }
        tma_load_3d(ring_w + st * kWBox, &p.wmap[map], 0, is_box * NC, row0, bar);
        tma_load_3d(ring_s + st * kSBox, &p.smap[map], 0, is_box * NC, srow, bar);
        ++issued;
        ++is_b;
        if (++is_box == nbox) {
            is_box = 0;
            if (++is_tile == tiles) {
                is_tile = 0;
                ++is_grp;
            }
        }
    };
    if constexpr (!MOE) {
        set_ranges(p.items_q);  // dense: items_q holds the number of jobs
        start_cursor();
        if (lane == 0)
            for (int s = 0; s < stages; ++s) issue_next();
        if (warp == tk::kWarps - 1 && lane < p.M) {
            const uint16_t* xr = p.x + static_cast<int64_t>(lane) * p.K;
            prefetch_l2_bulk(xr, static_cast<uint32_t>(p.K) * 2u);
            prefetch_l2(xr);
        }
    } else {
        if (warp == tk::kWarps - 1 && lane == 0) prefetch_l2(p.ids);
        const int xrows_all = p.x_per_slot ? p.slots : (p.slots + p.top_k - 1) / p.top_k;
        if (warp == tk::kWarps - 2 && lane < xrows_all)
            prefetch_l2_bulk(p.x + static_cast<int64_t>(lane) * p.K, static_cast<uint32_t>(p.K) * 2u);
    }
    if (tid == 0) trace_phase(p.trace_slot, 1);
    pdl_launch_dependents();
    pdl_wait();
    if (tid == 0) trace_phase(p.trace_slot, 2);

    int M = p.M;
    const int* rowsel = nullptr;
    bool x_overflow = false;  // the CTA computes in fp32 with x from global memory
    if constexpr (MOE) {
        // more than 32 slots: all threads build the groups, with scratch in the x region (free
        // until x is staged); each CTA then keeps only the groups of its own job range
        const bool big = p.slots > kTileMoeSlots;
        int* scratch = reinterpret_cast<int*>(sbase + p.x_off);
        if (big) tile_moe_groups_big(p, tab, scratch, tid);
        else if (warp == 0) tile_moe_groups(p, tab, lane);
        if (!big && tid == 0) trace_word(p.trace_slot, 38, static_cast<unsigned long long>(clock64()));
        __syncthreads();
        if (!big && tid == 0) trace_word(p.trace_slot, 39, static_cast<unsigned long long>(clock64()));
#if NVFP4_SK_GROUP_ALIGNED
        if (p.items_r) {
            // group-aligned: CTAs [G*g/ng, G*(g+1)/ng) share group g's jobs (the planner keeps
            // G >= the most groups there can be), so a CTA stages one group's x rows (<= 8)
            const int ng = tab->n_groups, G = static_cast<int>(gridDim.x), b = static_cast<int>(blockIdx.x);
            if (ng > 0) {
                // 32-bit unsigned arithmetic: b < G and ng <= kMaxMoeSlots keep (b + 1) * ng and
                // G * (g + 1) far below 2^32, and tiles * k (k <= c) too while tiles < 2^22 and
                // c <= 1024 (else 64-bit)
                const uint32_t ug = (static_cast<uint32_t>(b + 1) * static_cast<uint32_t>(ng) - 1u) /
                                    static_cast<uint32_t>(G);
                const int g = static_cast<int>(ug);
                const int lo = static_cast<int>(static_cast<uint32_t>(G) * ug / static_cast<uint32_t>(ng));
                const int c = static_cast<int>(static_cast<uint32_t>(G) * (ug + 1u) / static_cast<uint32_t>(ng)) - lo;
                const int i = b - lo;
                auto part = [&](int k) -> int {  // tiles * k / c
                    if (tiles < (1 << 22) && c <= 1024)
                        return static_cast<int>(static_cast<uint32_t>(tiles) * static_cast<uint32_t>(k) /
                                                static_cast<uint32_t>(c));
                    return static_cast<int>(static_cast<long long>(tiles) * k / c);
                };
                if (c > 0 && i >= 0 && i < c) {
                    j0 = g * tiles + part(i);
                    j1 = g * tiles + part(i + 1);
                } else {
                    // fewer CTAs than groups (the planner rules it out): no work, flagged
                    j0 = j1 = 0;
                    if (tid == 0) raise_status(NVFP4_DEV_INTERNAL, p.status_user);
                }
            } else {
                j0 = j1 = 0;
            }
            const int total = (j1 - j0) * nbox;
            bs = (warp * total) >> 3;
            be = ((warp + 1) * total) >> 3;
        } else {
            set_ranges(tab->n_groups * tiles);
        }
#else
        set_ranges(tab->n_groups * tiles);
#endif
        if (big) {
            if (j0 < j1 && (j1 - 1) / tiles - j0 / tiles + 1 > kMoeWindow) {
                // more groups than the window holds (the planner rules it out): no work, flagged
                if (tid == 0) raise_status(NVFP4_DEV_INTERNAL, p.status_user);
                j0 = j1 = 0;
                bs = be = 0;
            }
            tile_moe_window(p, tab, scratch, j0 < j1 ? j0 / tiles : 1, j0 < j1 ? (j1 - 1) / tiles : 0, tid);
        } else if (warp == 0 && j0 < j1) {
            tile_moe_rows(p, tab, j0 / tiles, (j1 - 1) / tiles, lane);
        }
        __syncthreads();
        gw0 = tab->g0;
        start_cursor();
        if constexpr (SD) {
            // dictionary scales: the planner keeps the CTA inside one group (group-aligned
            // ranges), so one pair table serves all of its jobs
            if (j0 < j1)
                build_pair_table(reinterpret_cast<uint32_t*>(sbase + p.sdtab_off),
                                 p.sd_dict + 32 * tab->expert[j0 / tiles - gw0], tid, tk::kThreads);
            if (tid == 0 && j0 < j1 && (j1 - 1) / tiles != j0 / tiles) raise_status(NVFP4_DEV_INTERNAL, p.status_user);
            __syncthreads();
        }
        M = j0 < j1 ? tab->nrows : 0;
        rowsel = tab->rows;
        if (M > p.M) {  // more x rows than the staging buffer holds (more than 32 slots only)
            x_overflow = true;
            M = 0;
        }
        if (tid == 0) trace_word(p.trace_slot, 36, static_cast<unsigned long long>(clock64()));
        if (lane == 0)
            for (int s = 0; s < min(stages, NVFP4_MOE_EARLY); ++s) issue_next();
    }

    // x, all of K, staged by all eight warps
    uint8_t* const xs = sbase + p.x_off;
    float* const e2 = reinterpret_cast<float*>(sbase + p.misc_off);
    uint32_t* const gmax = reinterpret_cast<uint32_t*>(sbase + p.misc_off + tk::kWarps * 32);
    bool lossy = false;
    float e2v = 1.f;
    bool staged = M == 0;
    if (M > 0) {
        if (NVFP4_STAGE_BULK)
            staged = stage_x_bulk(p.x, rowsel, M, p.K, 0, p.K, xs, p.sstride, gmax + 16,
                                  reinterpret_cast<uint64_t*>(gmax + 24), warp, tk::kWarps, 2, lane, p.wait_ns);
        else
            staged = stage_x_direct<NVFP4_SK_STAGE_PRE>(p.x, rowsel, M, p.K, 0, p.K, xs, p.sstride, gmax + 16,
                                                         warp, tk::kWarps, 2, lane, [] {});
    }
    if (!staged) {
        lossy = stage_x_slice(p.x, rowsel, M, p.K, 0, p.K, xs, p.sstride, e2, gmax, warp, tk::kWarps, 2, lane);
        e2v = e2[0];
    }
    if (tid == 0) trace_phase(p.trace_slot, 3);
    if constexpr (MOE) {
        if (lane == 0)
            for (int s = min(stages, NVFP4_MOE_EARLY); s < stages; ++s) issue_next();
    }
    if (tid == 0) trace_word(p.trace_slot, 37, static_cast<unsigned long long>(clock64()));
    const bool use_f32 = lossy || p.force_f32 || x_overflow;
    if (use_f32 && (M > 0 || x_overflow) && warp == 0 && lane == 0) atomicAdd(&g_fp32_fallbacks, 1ull);
    bool traced_first = false;

    const int g = lane >> 2;
    const int ra = tile_row_perm<NC>(g), rb = ra + 8;
    const int m0 = 2 * t;
    const float e2s = use_f32 ? 1.f : e2v;
    const uint64_t budget = p.wait_ns;
    bool dead = false;

    auto ncols_of = [&](int grp) -> int {
        if constexpr (MOE) return tab->count[grp - gw0];
        else return p.M;
    };
    auto gscale_of = [&](int grp) -> float {
        if constexpr (MOE) return __ldg(p.g_dev + tab->expert[grp - gw0]);
        else return p.g[grp];
    };
    auto out_at = [&](int grp, int m, int row) -> int64_t {
        if constexpr (MOE) return static_cast<int64_t>(tab->slot[grp - gw0][m]) * p.N + row;
        else return m * p.ldy + static_cast<int64_t>(grp) * p.N + row;
    };

    // walk this warp's boxes
    {
        int job = j0 + bs / nbox, kb = bs - (bs / nbox) * nbox;
        int grp = job / tiles, tile = job - grp * tiles;
        const int first_job = job;
        bool whole = kb == 0;  // this warp holds the current job's first box
        float d[4] = {0.f, 0.f, 0.f, 0.f};
        float dd[kTileChains][4];
#pragma unroll
        for (int c = 0; c < kTileChains; ++c)
#pragma unroll
            for (int i = 0; i < 4; ++i) dd[c][i] = 0.f;
        float first_rec[4] = {0.f, 0.f, 0.f, 0.f}, last_rec[4] = {0.f, 0.f, 0.f, 0.f};
        // global scales of the groups of this warp's first and last jobs, requested now so that
        // the load is not waited for at a job's end (other groups load theirs there)
        int gs_grp0 = grp, gs_grp1 = grp;
        float gs0 = 1.f, gs1 = 1.f;
        if (bs < be) {
            gs_grp1 = (j0 + (be - 1) / nbox) / tiles;
            gs0 = gscale_of(gs_grp0);
            gs1 = gscale_of(gs_grp1);
        }
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
        uint32_t xa = 0;
        auto set_x = [&]() {
            int col = min(g, max(M - 1, 0));
            if constexpr (MOE) col = tab->col[grp - gw0][min(g, ncols_of(grp) - 1)];
            xa = base + p.x_off + static_cast<uint32_t>(col) * p.sstride;
        };
        if (bs < be) set_x();
        for (int b = bs; b < be; ++b) {
            if (!dead) {
                const uint32_t st = cons_st;
                const uint32_t ph = cons_ph;
                if (!__all_sync(0xffffffffu, budget != 0 && mbar_wait(&bars[st], ph, budget))) {
                    dead = true;
                    raise_status(NVFP4_DEV_TIMEOUT, nullptr);
                } else {
                    if (NVFP4_PHASE_TRACE && lane == 0 && !traced_first) {
                        if (warp == 0) trace_phase(p.trace_slot, 4);
                        else trace_word(p.trace_slot, 24 + warp, global_ns());
                        traced_first = true;
                    }
                    if (!use_f32) {
                        tile_slot_mma<NC, SD>(ring_w + st * kWBox, ring_s + st * kSBox, xa, kb * NC * 2, ra, t, dd,
                                              base + p.sdtab_off);
                    } else {
                        const int* xrow = nullptr;
                        if constexpr (MOE) xrow = tab->xrow[grp - gw0];
                        tile_slot_f32<NC, SD>(ring_w + st * kWBox, ring_s + st * kSBox, p.x, xrow, p.K, ncols_of(grp),
                                              kb * NC, ra, t, acc, base + p.sdtab_off);
                    }
                    cons_advance();
                    __syncwarp();
                    if (lane == 0) issue_next();
                }
            }
            if (kb == nbox - 1 || b == be - 1) {
                // this warp's part of the job ends here
                if (use_f32) {
#pragma unroll
                    for (int i = 0; i < 16; ++i) {
                        acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 1);
                        acc[i] += __shfl_xor_sync(0xffffffffu, acc[i], 2);
                    }
#pragma unroll
                    for (int m = 0; m < 8; ++m) {
                        if (m == m0) { d[0] = acc[m]; d[2] = acc[8 + m]; }
                        if (m == m0 + 1) { d[1] = acc[m]; d[3] = acc[8 + m]; }
                    }
#pragma unroll
                    for (int i = 0; i < 16; ++i) acc[i] = 0.f;
                } else {
#pragma unroll
                    for (int c = 0; c < kTileChains; ++c)
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            d[i] += dd[c][i];
                            dd[c][i] = 0.f;
                        }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) d[i] *= e2s;
                const int ncols = ncols_of(grp);
                if (whole && kb == nbox - 1) {
                    const float gs = grp == gs_grp0 ? gs0 : (grp == gs_grp1 ? gs1 : gscale_of(grp));
                    const int rowa = tile * 16 + ra, rowb = tile * 16 + rb;
                    if (m0 < ncols) {
                        if (rowa < p.N) store_out(p.y, out_at(grp, m0, rowa), d[0] * gs, p.out_bf16);
                        if (rowb < p.N) store_out(p.y, out_at(grp, m0, rowb), d[2] * gs, p.out_bf16);
                    }
                    if (m0 + 1 < ncols) {
                        if (rowa < p.N) store_out(p.y, out_at(grp, m0 + 1, rowa), d[1] * gs, p.out_bf16);
                        if (rowb < p.N) store_out(p.y, out_at(grp, m0 + 1, rowb), d[3] * gs, p.out_bf16);
                    }
                } else if (job == first_job) {
#pragma unroll
                    for (int i = 0; i < 4; ++i) first_rec[i] = d[i];  // written once the ring is idle
                } else {
#pragma unroll
                    for (int i = 0; i < 4; ++i) last_rec[i] = d[i];
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) d[i] = 0.f;
                // next job
                kb = 0;
                whole = true;
                ++job;
                if (++tile == tiles) {
                    tile = 0;
                    ++grp;
                }
                if (b + 1 < be) set_x();
            } else {
                ++kb;
            }
        }
        if (lane == 0) trace_word(p.trace_slot, 16 + warp, global_ns());
        if (tid == 0) trace_phase(p.trace_slot, 5);
        // the ring is idle once every issued copy has landed (only a timed-out warp has any left)
        if (lane == 0) {
            while (consumed < issued) {
                mbar_wait(&bars[cons_st], cons_ph, kDrainWaitNs);
                cons_advance();
            }
        }
        __syncwarp();
        float* r0 = rec_of(warp, 0);
        float* r1 = rec_of(warp, 1);
        r0[ra * 8 + m0] = first_rec[0];
        r0[ra * 8 + m0 + 1] = first_rec[1];
        r0[rb * 8 + m0] = first_rec[2];
        r0[rb * 8 + m0 + 1] = first_rec[3];
        r1[ra * 8 + m0] = last_rec[0];
        r1[ra * 8 + m0 + 1] = last_rec[1];
        r1[rb * 8 + m0] = last_rec[2];
        r1[rb * 8 + m0 + 1] = last_rec[3];
    }
    named_bar_sync(1, tk::kThreads);
    // jobs split between warps: the warp holding a job's first box adds the records in order
    if (bs < be) {
        const int jf = j0 + bs / nbox, jl = j0 + (be - 1) / nbox;
        for (int s = 0; s < 2; ++s) {
            const int j = s == 0 ? jf : jl;
            if (s == 1 && jl == jf) break;
            const int jb = (j - j0) * nbox, je = jb + nbox;  // the job's boxes in CTA units
            if (jb < bs) continue;                          // starts in an earlier warp
            if (jb >= bs && je <= be) continue;             // whole: stored already
            const int grp = j / tiles, tile = j - (j / tiles) * tiles;
            const int ncols = ncols_of(grp);
            const float gs = gscale_of(grp);
            for (int i = lane; i < 16 * ncols; i += 32) {
                const int r = i / ncols, m = i - r * ncols;
                float sum = rec_of(warp, s)[r * 8 + m];
                for (int w = warp + 1; w < tk::kWarps; ++w) {
                    const int wbs = (w * (j1 - j0) * nbox) >> 3, wbe = ((w + 1) * (j1 - j0) * nbox) >> 3;
                    if (wbs >= je) break;
                    if (wbe > wbs) sum += rec_of(w, 0)[r * 8 + m];  // the job is that warp's first one
                }
                const int row = tile * 16 + r;
                if (row < p.N) store_out(p.y, out_at(grp, m, row), sum * gs, p.out_bf16);
            }
        }
    }
    if (tid == 0) trace_phase(p.trace_slot, 6);
    if (lane == 0) {
        while (consumed < issued) {
            mbar_wait(&bars[cons_st], cons_ph, kDrainWaitNs);
            cons_advance();
        }
    }
    __syncwarp();
    if (tid == 0) trace_phase(p.trace_slot, 7);
    trace_flush(p.trace_slot, tid);
}

// ------------------------------------------------------------------ byte-load kernel

struct SimpleParams {
    const uint8_t* w[2];
    const uint8_t* s[2];
    float g[2];
    const float* g_dev;
    const int32_t* ids;
    int32_t* status_user;
    const uint16_t* x;
    void* y;
    int64_t ldy;
    int out_bf16;
    int M, N, K, groups;
    int moe, E, top_k, x_per_slot, slots;
    int swiglu;               // groups == 2: one output silu(clamp(gate)) * clamp(up) per column
    float clamp;
    int sd;                   // 1: s[] are dictionary index planes (dense: one; MoE: one per expert)
    const uint8_t* sd_dict;   // their tables: [32] (dense) or [E][32] (MoE)
};

// One warp per output column (all M rows). Lanes stride over the 16-element blocks of K.
template <int MT>
__global__ void __launch_bounds__(kSimpleThreads) gemv_simple_kernel(const __grid_constant__ SimpleParams p) {
    const int lane = threadIdx.x & 31;
    const int64_t col = static_cast<int64_t>(blockIdx.x) * (kSimpleThreads / 32) + (threadIdx.x >> 5);
    const int64_t Kh = p.K / 2, Ks = p.K / 16;
    const uint8_t* wrow;
    const uint8_t* srow;
    float g;
    int64_t xrow0 = 0;
    int64_t out0, out_step;
    int mrows = p.M;
    int64_t sd_row = 0;                  // dictionary scales: row of the index plane at srow
    const uint8_t* sd_tab = p.sd_dict;   // and its table
    if (p.moe) {
        if (col >= static_cast<int64_t>(p.slots) * p.N) return;
        const int sl = static_cast<int>(col / p.N);
        const int64_t n = col - static_cast<int64_t>(sl) * p.N;
        const int e = __ldg(p.ids + sl);
        if (e < 0 || e >= p.E) {
            if (lane == 0) {
                store_out(p.y, sl * p.ldy + n, 0.f, p.out_bf16);
                raise_status(NVFP4_DEV_BAD_EXPERT, p.status_user);
            }
            return;
        }
        wrow = p.w[0] + (static_cast<int64_t>(e) * p.N + n) * Kh;
        srow = p.s[0] + (static_cast<int64_t>(e) * p.N + n) * Ks;
        if (p.sd) {
            srow = p.s[0] + e * sd_plane_bytes(p.N, p.K);
            sd_row = n;
            sd_tab = p.sd_dict + 32 * e;
        }
        g = __ldg(p.g_dev + e);
        xrow0 = p.x_per_slot ? sl : sl / p.top_k;
        out0 = sl * p.ldy + n;
        out_step = 0;
        mrows = 1;
    } else {
        const int64_t cols = p.swiglu ? p.N : static_cast<int64_t>(p.groups) * p.N;
        if (col >= cols) return;
        const int grp = p.swiglu ? 0 : static_cast<int>(col / p.N);
        const int64_t n = col - static_cast<int64_t>(grp) * p.N;
        wrow = p.w[grp] + n * Kh;
        srow = p.s[grp] + n * Ks;
        g = p.g[grp];
        if (p.sd) {
            srow = p.s[grp];
            sd_row = n;
        }
        out0 = col;
        out_step = p.ldy;
    }
    // acc[m] = sum over K of the row's products with x row xrow0 + m, summed over the warp
    auto dot = [&](const uint8_t* wr, const uint8_t* sr, float (&acc)[MT]) {
#pragma unroll
        for (int m = 0; m < MT; ++m) acc[m] = 0.f;
        for (int64_t b = lane; b < Ks; b += 32) {
            const uint32_t code = p.sd ? sd_code(sr, sd_tab, p.K, sd_row, b) : __ldg(sr + b);
            const uint32_t shf = cvt_e4m3x2(static_cast<uint16_t>(code));
            const uint16_t sc = static_cast<uint16_t>(shf & 0xffffu);
            for (int e = 0; e < 8; ++e) {
                uint32_t h[4];
                cvt_e2m1x8(static_cast<uint32_t>(__ldg(wr + b * 8 + e)), h);
                const float2 q = widen_scaled(h[0], sc);
                const int64_t k = b * 16 + 2 * e;
#pragma unroll
                for (int m = 0; m < MT; ++m) {
                    if (m < mrows) {
                        const uint16_t* xr = p.x + (xrow0 + m) * p.K + k;
                        const float x0 = __uint_as_float(static_cast<uint32_t>(__ldg(xr)) << 16);
                        const float x1 = __uint_as_float(static_cast<uint32_t>(__ldg(xr + 1)) << 16);
                        acc[m] = fmaf(q.x, x0, acc[m]);
                        acc[m] = fmaf(q.y, x1, acc[m]);
                    }
                }
            }
        }
#pragma unroll
        for (int m = 0; m < MT; ++m) {
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) acc[m] += __shfl_xor_sync(0xffffffffu, acc[m], o);
        }
    };
    float acc[MT];
    dot(wrow, srow, acc);
    if (!p.moe && p.swiglu) {
        // the same column of the up projection, then the fused activation
        float accu[MT];
        dot(p.w[1] + col * Kh, p.s[1] + col * Ks, accu);
        if (lane == 0) {
#pragma unroll
            for (int m = 0; m < MT; ++m)
                if (m < mrows)
                    store_out(p.y, out0 + m * out_step, swiglu_f32(g * acc[m], p.g[1] * accu[m], p.clamp),
                              p.out_bf16);
        }
        return;
    }
    if (lane == 0) {
#pragma unroll
        for (int m = 0; m < MT; ++m)
            if (m < mrows) store_out(p.y, out0 + m * out_step, g * acc[m], p.out_bf16);
    }
}

// ------------------------------------------------------------------ host side

struct DeviceInfo {
    int sm_count = 0;
    int smem_optin = 0;   // per block
    int smem_per_sm = 0;
    bool init = false;
};

std::mutex g_mu;
DeviceInfo g_dev[64];
uint64_t g_wait_ns = kDefaultWaitNs;
// Kernel selection; NVFP4_GEMV_FORCE_VARIANT=0..3 in the environment sets the initial value
// (for tests and benchmarks), nvfp4_set_variant changes it.
int initial_variant() {
    const char* v = std::getenv("NVFP4_GEMV_FORCE_VARIANT");
    if (!v || !*v) return 0;
    char* end = nullptr;
    const long n = std::strtol(v, &end, 10);
    return (end && *end == '\0' && n >= 0 && n <= 3) ? static_cast<int>(n) : 0;
}
int g_variant = initial_variant();
int g_last_cuda_error = 0;

const DeviceInfo* device_info(int* dev_out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return nullptr;
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (!d.init) {
        if (cudaDeviceGetAttribute(&d.sm_count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return nullptr;
        if (cudaDeviceGetAttribute(&d.smem_optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
            return nullptr;
        if (cudaDeviceGetAttribute(&d.smem_per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess)
            return nullptr;
        d.init = true;
    }
    if (dev_out) *dev_out = dev;
    return &d;
}

nvfp4_status cuda_fail(cudaError_t e) {
    g_last_cuda_error = static_cast<int>(e);
    return NVFP4_ERR_CUDA;
}

struct Plan {
    int kind;      // 0 stream dense, 1 stream MoE, 2 simple
    int mt;
    Params p;
    int grid;
    uint32_t smem;
};

bool g_pdl = true;

uint32_t align_up(uint32_t v, uint32_t a) { return (v + a - 1) / a * a; }

// Bytes between weight rows in a ring slot: rows are stored as they sit in HBM, so one bulk
// copy moves a whole item (S == 1).
int padded_wstride(int Kr) { return Kr / 2; }

// Shared-memory layout and counts for a K range; false if it does not fit.
// n_units = CTAs (S == 1) or clusters (S > 1) that share the items.
bool layout(Params& p, int mt, int rows_total_est, int groups_for_items, int n_units, int smem_limit,
            uint32_t* smem_out) {
    const int R = kTileRows;
    p.wstride = padded_wstride(p.Kr);
    const int srow = p.S == 1 ? p.K / 16 : p.Kr / 16;
    const int row_bytes = p.wstride + srow;
    const int rpi_cap = kStageData / row_bytes;
    if (rpi_cap < 1) return false;
    // Rows per item: the value that minimises, for the busiest unit, the row slots it
    // decodes (a partial 16-row MMA tile still costs 16) plus the rows it streams plus a
    // per-item overhead, preferring larger items on ties.
    int best_rpi = 1;
    long long best_rows_cost = -1;
    for (int rpi = 1; rpi <= rpi_cap; ++rpi) {
        const long long items = static_cast<long long>(groups_for_items) * ((p.N + rpi - 1) / rpi);
        const long long per_unit = (items + n_units - 1) / n_units;
        const long long slots = rpi <= 8 ? 8 : (rpi + R - 1) / R * R;  // a tile with <= 8 rows decodes half
        const long long cost = per_unit * (slots + rpi + 2);  // decode slots + streamed rows + per-item work
        if (best_rows_cost < 0 || cost <= best_rows_cost) { best_rows_cost = cost; best_rpi = rpi; }
    }
    const int rpi = best_rpi;
    p.rpi = rpi;
    p.chunks = (p.N + rpi - 1) / rpi;
    p.items = groups_for_items * p.chunks;
    p.J = (p.Kr + kStepElems - 1) / kStepElems;
    p.work = static_cast<long long>((p.items + n_units - 1) / n_units) * ((rpi <= 8 ? 8 : (rpi + R - 1) / R * R) + rpi + 2) * p.Kr;
    if (p.S > 1) p.work += p.work / 2;  // per-row copies, cluster reduction and co-scheduling
    const int items_per_unit = (p.items + n_units - 1) / n_units;
    // warps along K: fewest passes over (16-row tiles x 128-element steps); ties go to fewer
    const int steps = (p.Kr + 127) / 128, tiles = (rpi + R - 1) / R;
    int best_ck = 1, best_cost = 1 << 30;
    for (int ck = 1; ck <= kConsumerWarps; ck *= 2) {
        const int cr = kConsumerWarps / ck;
        const int cost = ((steps + ck - 1) / ck) * ((tiles + cr - 1) / cr);
        if (cost < best_cost) { best_cost = cost; best_ck = ck; }
    }
    p.ck = best_ck;
    p.cr = kConsumerWarps / best_ck;
    p.mstride = mt;
    p.xh_stride = steps * 256 + 64;
    p.stage_stride = align_up(static_cast<uint32_t>(rpi) * row_bytes + 128, 128);
    // a CTA with at most two items needs no deeper ring; otherwise the deepest ring that fits
    for (int stages = items_per_unit <= 2 ? 2 : kMaxStages; stages >= 2; --stages) {
        p.stages = stages;
        uint32_t off = static_cast<uint32_t>(p.stages) * p.stage_stride;
        p.x_off = off;
        off += align_up(static_cast<uint32_t>(mt) * p.xh_stride, 128);
        p.xraw_off = off;
        off += align_up(static_cast<uint32_t>(mt) * p.Kr * 2, 128);
        p.misc_off = off;
        off += align_up((8 + 16 * kConsumerWarps) * 4, 128);
        p.red_off = off;
        uint32_t red_bytes = static_cast<uint32_t>(p.stages) * p.ck * rpi * mt * 4;
        const uint32_t moe_scratch = 3 * kMaxMoeSlots * 4;
        if (red_bytes < moe_scratch) red_bytes = moe_scratch;  // MoE table build reuses it
        off += align_up(red_bytes, 128);
        p.cl_off = off;
        if (p.S > 1) {
            p.cl_rows = items_per_unit * rpi;
            off += align_up(static_cast<uint32_t>(p.cl_rows) * mt * 4, 128);
        } else {
            p.cl_rows = 0;
        }
        p.tab_off = off;
        off += align_up(sizeof(MoeTables), 128);
        p.bar_off = off;
        off += kNumBars * 8 + 16;
        *smem_out = off;
        if (off <= static_cast<uint32_t>(smem_limit)) return true;
    }
    return false;
}

// Dense / gate-up plan. groups = 1 (dense) or 2 (gate_up).
bool plan_dense(Plan& pl, int M, int N, int K, int groups, const DeviceInfo& d, const uint8_t* const* w,
                const uint8_t* const* s, const void* x) {
    if (g_variant == 1) return false;
    if (K % 32 != 0 || (reinterpret_cast<uintptr_t>(x) & 15)) return false;  // x rows are bulk-copied
    for (int i = 0; i < groups; ++i)
        if ((reinterpret_cast<uintptr_t>(w[i]) & 15) || (reinterpret_cast<uintptr_t>(s[i]) & 1)) return false;
    const int mt = M;
    // Try every K split; keep the one whose busiest unit decodes the fewest row-elements
    // (partial 16-row tiles included), the smaller split on ties. Two CTAs per SM when two
    // rings fit, so their decoding warps hide each other's latencies.
    bool found = false;
    for (int S = 1; S <= 8; ++S) {
        if (S > 1 && (K % (256 * S) != 0)) continue;
        Params p{};
        uint32_t smem = 0;
        int n_units = 0;
        bool ok = false;
        for (int per_sm = (S == 1 ? 2 : 1); per_sm >= 1 && !ok; --per_sm) {
            p = Params{};
            p.M = M; p.N = N; p.K = K; p.groups = groups; p.S = S; p.Kr = K / S;
            n_units = S == 1 ? d.sm_count * per_sm : d.sm_count / S;
            const int limit = per_sm == 1 ? d.smem_optin : d.smem_per_sm / per_sm - 1024;
            ok = n_units >= 1 && layout(p, mt, groups * N, groups, n_units, limit, &smem);
            if (ok && per_sm == 2) p.work /= 2;  // two units share one SM's time
        }
        if (n_units < 1) break;
        if (!ok) continue;
        if (found && p.work >= pl.p.work) continue;
        const int units = std::min(n_units, p.items);
        p.items_q = p.items / units;
        p.items_r = p.items - p.items_q * units;
        p.s_aligned = K % 256 == 0;
        for (int i = 0; i < groups; ++i) p.s_aligned &= (reinterpret_cast<uintptr_t>(s[i]) & 15) == 0;
        pl.kind = 0;
        pl.mt = mt;
        pl.p = p;
        pl.grid = units * S;
        pl.smem = smem;
        found = true;
    }
    return found;
}

bool plan_moe(Plan& pl, int E, int T, int top_k, int N, int K, const DeviceInfo& d, const uint8_t* w,
              const uint8_t* s, const void* x) {
    if (g_variant == 1) return false;
    if (reinterpret_cast<uintptr_t>(x) & 15) return false;  // x rows are bulk-copied
    const int slots = T * top_k;
    if (slots > kMaxMoeSlots || K % 32 != 0) return false;
    if ((reinterpret_cast<uintptr_t>(w) & 15) || (reinterpret_cast<uintptr_t>(s) & 1)) return false;
    // largest member cap that fits two CTAs per SM, else one CTA per SM
    const int caps[4] = {8, 4, 2, 1};
    for (int per_sm = 2; per_sm >= 1; --per_sm) {
        for (int ci = 0; ci < 4; ++ci) {
            const int mt = caps[ci];
            if (mt > slots && mt > 1) continue;
            Params p{};
            p.N = N; p.K = K; p.S = 1; p.Kr = K; p.E = E; p.T = T; p.top_k = top_k; p.slots = slots;
            uint32_t smem = 0;
            const int limit = per_sm == 1 ? d.smem_optin : d.smem_per_sm / per_sm - 1024;
            if (!layout(p, mt, slots * N, slots, d.sm_count * per_sm, limit, &smem)) continue;
            p.s_aligned = K % 256 == 0 && (reinterpret_cast<uintptr_t>(s) & 15) == 0;
            pl.kind = 1;
            pl.mt = mt;
            pl.p = p;
            pl.grid = d.sm_count * per_sm;  // the item count depends on the routing, known on the device
            pl.smem = smem;
            return true;
        }
    }
    return false;
}

// Raises a kernel's dynamic shared-memory limit to the device maximum once per device and
// kernel (`done` belongs to the caller's instantiation), so launches with different plans
// never change the attribute again.
template <typename Kern>
cudaError_t allow_max_smem(Kern kern, bool (&done)[64]) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lk(g_mu);
    if (!done[dev]) {
        // the opt-in limit covers static and dynamic shared memory together
        cudaFuncAttributes fa{};
        e = cudaFuncGetAttributes(&fa, kern);
        if (e != cudaSuccess) return e;
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 g_dev[dev].smem_optin - static_cast<int>(fa.sharedSizeBytes));
        if (e != cudaSuccess) return e;
        done[dev] = true;
    }
    return cudaSuccess;
}

template <int MODE, int MT>
cudaError_t launch_stream(const Plan& pl, cudaStream_t st) {
    auto kern = gemv_stream_kernel<MODE, MT>;
    static bool done[64] = {};
    cudaError_t e = allow_max_smem(kern, done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(pl.grid);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = pl.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (pl.p.S > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = pl.p.S;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (g_pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, pl.p);
}

cudaError_t dispatch_stream(const Plan& pl, cudaStream_t st) {
    if (pl.kind == 1) {
        switch (pl.mt) {
            case 1: return launch_stream<kModeMoe, 1>(pl, st);
            case 2: return launch_stream<kModeMoe, 2>(pl, st);
            case 4: return launch_stream<kModeMoe, 4>(pl, st);
            case 8: return launch_stream<kModeMoe, 8>(pl, st);
            default: return cudaErrorInvalidValue;
        }
    }
    switch (pl.mt) {
        case 1: return launch_stream<kModeDense, 1>(pl, st);
        case 2: return launch_stream<kModeDense, 2>(pl, st);
        case 3: return launch_stream<kModeDense, 3>(pl, st);
        case 4: return launch_stream<kModeDense, 4>(pl, st);
        case 5: return launch_stream<kModeDense, 5>(pl, st);
        case 6: return launch_stream<kModeDense, 6>(pl, st);
        case 7: return launch_stream<kModeDense, 7>(pl, st);
        case 8: return launch_stream<kModeDense, 8>(pl, st);
        default: return cudaErrorInvalidValue;
    }
}

// ------------------------------------------------------------------ tile kernel: host side

// Build-time planner overrides for tuning experiments (0 = let the cost model choose).
#ifndef NVFP4_TILE_KSPLIT
#define NVFP4_TILE_KSPLIT 0
#endif
#ifndef NVFP4_TILE_NC
#define NVFP4_TILE_NC 0
#endif
#ifndef NVFP4_TILE_S
#define NVFP4_TILE_S 0
#endif
#ifndef NVFP4_TILE_PER_SM
#define NVFP4_TILE_PER_SM 0  // nonzero: dense launches use at most this many CTAs per SM
#endif

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    });
    return fn;
}

// Groups a routing of T tokens to top_k distinct experts each, out of E, is expected to
// form when the experts are uniform: the expected number of distinct experts (each with at
// most 8 slots, so one group each), E * (1 - (1 - top_k / E)^T), rounded, at least 1.
int expected_groups(int E, int T, int top_k) {
    if (E <= 0 || T <= 0 || top_k <= 0) return 1;
    const double q = 1.0 - std::min(1.0, static_cast<double>(top_k) / E);
    double miss = 1.0;
    for (int i = 0; i < T; ++i) miss *= q;
    const double g = E * (1.0 - miss);
    return std::max(1, std::min(T * top_k, static_cast<int>(g + 0.5)));
}

struct TilePlan {
    TileParams p;
    int nc;
    int grid_x, grid_y;  // SM slots x CTAs per slot
    uint32_t smem;
    bool sk;             // stream-K form (gemv_tile_sk_kernel)
};

// Tile-kernel plan for a dense (groups = 1) or gate/up (groups = 2) call; false when the
// call does not meet the kernel's preconditions or its x does not fit next to the rings.
// The cost of a candidate is the larger of a latency term (rounds of items a CTA runs times
// the 128-element steps of one warp per item) and a throughput term (items on the busiest
// SM times the steps each of its warps decodes), both in units of one warp step.
bool plan_tile(TilePlan& tp, int M, int N, int K, int groups, const DeviceInfo& d, const uint8_t* const* w,
               const uint8_t* const* s, const void* x, bool moe = false, int moe_rows = 0, int moe_groups_max = 0,
               bool swiglu = false, bool need_encoder = true, bool sd = false, double* cost_out = nullptr) {
    if (g_variant == 1 || g_variant == 3) return false;
    if (sd && (swiglu || (!moe && groups != 1))) return false;  // dictionary scales: dense or MoE
    // scale box per ring slot and the pair table (dictionary scales)
    auto sbox = [&](int nc) -> uint32_t {
        return sd ? (nc == 2 ? scale_box_bytes<2, true>() : scale_box_bytes<1, true>()) : static_cast<uint32_t>(nc) * 256u;
    };
    const uint32_t sdtab = sd ? kSdPairs * 4u : 0u;
    if (K <= 0 || K % 256 != 0 || M < 1 || M > 8 || N < 1 || N > (1 << 27)) return false;
    // MoE: M is the largest number of columns of a group (8), groups the expected number of
    // groups (cost only), moe_groups_max the most there can be; moe_rows x rows exist in all
    const int xrows = moe ? moe_rows : M;
    if (reinterpret_cast<uintptr_t>(x) & 15) return false;
    const int tensors = moe ? 1 : groups;  // weight tensors: one for all experts, else one per group
    for (int i = 0; i < tensors; ++i)
        if ((reinterpret_cast<uintptr_t>(w[i]) & 15) || (reinterpret_cast<uintptr_t>(s[i]) & 15)) return false;
    if (need_encoder && !tensor_map_encoder()) return false;
    const int segs = K / 256;
    // gate/up with the fused activation: one group of 2 * tiles, gate and up tiles alternating,
    // so that an item (an even number of tiles) holds whole pairs
    const int tiles = swiglu ? 2 * ((N + 15) / 16) : (N + 15) / 16;
    const int item_groups = swiglu ? 1 : groups;
    bool found = false;
    double best = 0.0;
    for (int nc = 2; nc >= 1; --nc) {
        if (segs % nc) continue;
        const int nbox = segs / nc;
        for (int sl = 0; (1 << sl) <= 8; ++sl) {
            const int S = 1 << sl;
            // MoE with dictionary scales or more than 32 slots: stream-K only
            if (S > nbox || (moe && S > 1) || (moe && sd) || (moe && moe_groups_max > kTileMoeSlots)) break;
            if (NVFP4_TILE_S && S != NVFP4_TILE_S) continue;
            const int nbs = (nbox + S - 1) / S;  // most boxes of one rank
            for (int lg = 0; (1 << lg) <= tk::kWarps; ++lg) {
                const int ksplit = 1 << lg;
                if (S * ksplit > nbox) break;
                if (NVFP4_TILE_KSPLIT && ksplit != NVFP4_TILE_KSPLIT) continue;
                if (NVFP4_TILE_NC && nc != NVFP4_TILE_NC) continue;
                const int tpi = tk::kWarps / ksplit;
                if (swiglu && tpi < 2) continue;
                const int ipg = (tiles + tpi - 1) / tpi;
                const long long items = static_cast<long long>(item_groups) * ipg;
                if (items > (1LL << 30)) continue;
                const int nbmax = (nbs + ksplit - 1) / ksplit;  // most boxes of one warp per item
                const uint32_t sstride = static_cast<uint32_t>(nbmax) * nc * 512u + 64u;
                int rows_cap = xrows;
                if (moe) {
                    // the launch has units >= min(SMs, items) (items: the expected count), so a
                    // unit runs at most ipu contiguous items of the largest possible count, and
                    // touches at most ceil(ipu / ipg) + 1 groups of at most 8 columns each
                    const long long items_max = static_cast<long long>(std::max(moe_groups_max, groups)) * ipg;
                    const long long units_lo = std::min<long long>(d.sm_count, items);
                    const long long ipu = (items_max + units_lo - 1) / units_lo;
                    const long long span = (ipu + ipg - 1) / ipg + 1;
                    rows_cap = static_cast<int>(std::min<long long>(xrows, 8 * span));
                }
                const uint32_t x_bytes = align_up(static_cast<uint32_t>(ksplit * rows_cap) * sstride, 128);
                // deepest ring that still allows two CTAs per SM, else the deepest that fits one
                int stages = 0, per_sm = 0;
                uint32_t smem = 0;
                TileParams lp{};
                for (int want = 2; want >= 1 && !stages; --want) {
                    for (int st = tk::kMaxStages; st >= 2; --st) {
                        TileParams q{};
                        uint32_t off = 0;
                        q.ring_w = off;
                        off += static_cast<uint32_t>(tk::kWarps * st * nc) * 2048u;
                        q.ring_s = off;
                        off += static_cast<uint32_t>(tk::kWarps * st) * sbox(nc);
                        q.sdtab_off = off;
                        off += sdtab;
                        q.x_off = off;
                        off += x_bytes;
                        q.red_off = off;
                        if (ksplit > 1) off += 2u * tk::kRedFloats * 4u;
                        q.cpart_off = off;
                        if (S > 1 || swiglu) off += 2u * tk::kWarps * 16 * 8 * 4u;
                        q.misc_off = off;
                        off += align_up(tk::kWarps * 32 + tk::kWarps * 32 * 4, 128);  // e2, extremes, votes
                        q.bar_off = off;
                        off += tk::kWarps * tk::kMaxStages * 8;
                        q.moe_off = align_up(off, 16);
                        if (moe) off = q.moe_off + static_cast<uint32_t>(sizeof(TileMoe));
                        const uint32_t total = off + 1024;  // slack to align the base to 1024 bytes
                        const uint32_t limit = want == 2 ? static_cast<uint32_t>(d.smem_per_sm / 2 - 1024)
                                                         : static_cast<uint32_t>(d.smem_optin);
                        if (total <= limit) {
                            stages = st;
                            per_sm = want;
                            smem = total;
                            lp = q;
                            break;
                        }
                    }
                }
                if (!stages) continue;
                // Cost in units of one warp's 128-element step: the larger of a latency term (the
                // items one unit runs in sequence, each with its steps, reductions and barriers)
                // and a throughput term (all warp steps spread over the SMs at 16 warps each),
                // plus the staging of x, which shrinks with the K range of one CTA.
                const int per_sm_cap = (NVFP4_TILE_PER_SM && !moe) ? std::min(per_sm, NVFP4_TILE_PER_SM) : per_sm;
                const long long max_units = std::max<long long>(1, static_cast<long long>(d.sm_count) * per_sm_cap / S);
                const long long units = std::min(items, max_units);
                const long long ipu = (items + units - 1) / units;
                // (MoE, compared with the stream-K form: each box also costs about half a step of
                // wait, re-issue and loop)
                const double spw = 2.0 * nc * nbmax + (moe ? 0.5 * nbmax : 0.0);
                // measured: a reduction over warps costs ~2 steps, one over a cluster ~10
                const double ovh = (ksplit > 1 ? (moe ? 4.0 : 2.0) : 0.3) + (S > 1 ? 10.0 : 0.0);
                const double lat = static_cast<double>(ipu) * (spw + ovh);
                const double thr = static_cast<double>(items) * tk::kWarps * S * spw / (d.sm_count * 16.0) * 1.1;
                const double stage = static_cast<double>(moe ? std::min(rows_cap, 8) : xrows) * K / (2048.0 * S);
                const double cost = std::max(lat, thr) + stage;
                if (!found || cost < best - 1e-9) {
                    found = true;
                    best = cost;
                    tp.p = lp;
                    tp.p.M = rows_cap;
                    tp.p.N = N;
                    tp.p.K = K;
                    tp.p.tiles = tiles;
                    tp.p.ksplit_log2 = lg;
                    tp.p.s_log2 = sl;
                    tp.p.tpi = tpi;
                    tp.p.ipg = ipg;
                    tp.p.items_q = static_cast<int>(items / units);
                    tp.p.items_r = static_cast<int>(items % units);
                    tp.p.nbox = nbox;
                    tp.p.stages = stages;
                    tp.p.sstride = sstride;
                    tp.nc = nc;
                    tp.grid_x = static_cast<int>(units) * S;
                    tp.grid_y = 1;
                    tp.smem = smem;
                    tp.sk = false;
                }
            }
        }
    }
    // Stream-K form (MoE): whole K per CTA, jobs (group, tile) split evenly over the CTAs and
    // boxes evenly over the warps. Many jobs per CTA make it balance far better than items.
    if (moe && NVFP4_TILE_KSPLIT == 0 && NVFP4_TILE_S == 0) {
        for (int nc = 2; nc >= 1; --nc) {
            if (segs % nc || (NVFP4_TILE_NC && nc != NVFP4_TILE_NC)) continue;
            const int nbox = segs / nc;
            const long long jobs = static_cast<long long>(groups) * tiles;
            if (jobs > (1LL << 30) || jobs * nbox > (1LL << 30)) continue;
            const uint32_t sstride = static_cast<uint32_t>(K) * 2u + 64u;
            const long long jobs_max = static_cast<long long>(std::max(moe_groups_max, groups)) * tiles;
            const long long units_lo = std::min<long long>(d.sm_count, jobs);
            const long long jpc_max = (jobs_max + units_lo - 1) / units_lo;
          // (dictionary scales need group-aligned ranges: one pair table per CTA)
          for (int aligned = sd ? 1 : 0; aligned <= NVFP4_SK_GROUP_ALIGNED; ++aligned) {
            // aligned: every CTA inside one group, so at most 8 staged rows; needs a CTA per
            // group at least, whatever the routing
            const int groups_most = std::max(moe_groups_max, groups);
            // groups one CTA's job range can touch: more than 32 slots keep them in a window of
            // kMoeWindow table entries, and build the groups in the x region (5 KB of scratch).
            // Their staging buffer holds 8 x rows, a window's rows for the usual routings (an
            // expert has a few slots); a CTA whose window needs more computes in exact fp32
            // with x read from global memory instead.
            const long long span = aligned ? 1 : (jpc_max + tiles - 1) / tiles + 1;
            const bool big = moe_groups_max > kTileMoeSlots;
            if (big && span > kMoeWindow) continue;
            const int rows_cap = static_cast<int>(std::min<long long>(xrows, big ? 8 : 8 * span));
            uint32_t x_bytes = align_up(static_cast<uint32_t>(rows_cap) * sstride, 128);
            if (big) x_bytes = std::max<uint32_t>(x_bytes, kMoeScratchInts * 4u);
            int stages = 0, per_sm = 0;
            uint32_t smem = 0;
            TileParams lp{};
            for (int want = 2; want >= 1 && !stages; --want) {
                for (int st = tk::kMaxStages; st >= 2; --st) {
                    TileParams q{};
                    uint32_t off = 0;
                    q.ring_w = off;
                    off += static_cast<uint32_t>(tk::kWarps * st * nc) * 2048u;
                    q.ring_s = off;
                    off += static_cast<uint32_t>(tk::kWarps * st) * sbox(nc);
                    q.sdtab_off = off;
                    off += sdtab;
                    q.x_off = off;
                    off += x_bytes;
                    q.red_off = off;  // unused: partial records live in the drained rings
                    q.cpart_off = off;
                    q.misc_off = off;
                    off += align_up(tk::kWarps * 32 + tk::kWarps * 32 * 4, 128);
                    q.bar_off = off;
                    off += tk::kWarps * tk::kMaxStages * 8;
                    q.moe_off = align_up(off, 16);
                    off = q.moe_off + static_cast<uint32_t>(sizeof(TileMoe));
                    const uint32_t total = off + 1024;
                    const uint32_t limit = want == 2 ? static_cast<uint32_t>(d.smem_per_sm / 2 - 1024)
                                                     : static_cast<uint32_t>(d.smem_optin);
                    if (total <= limit) {
                        stages = st;
                        per_sm = want;
                        smem = total;
                        lp = q;
                        break;
                    }
                }
            }
            if (!stages) continue;
            long long units = std::min<long long>(jobs, static_cast<long long>(d.sm_count) * per_sm);
            long long jpc = (jobs + units - 1) / units;
            if (aligned) {
                units = static_cast<long long>(d.sm_count) * per_sm;
                if (units < groups_most) continue;
                const long long per_group = units / std::max(groups, 1);  // CTAs of the smallest share
                jpc = (tiles + per_group - 1) / per_group;
            }
            const double boxes_per_warp = static_cast<double>((jpc * nbox + tk::kWarps - 1) / tk::kWarps);
            const double lat = boxes_per_warp * (2.0 * nc + 0.5) + 2.0;
            const double thr = static_cast<double>(jobs) * nbox * (2.0 * nc + 0.5) / (d.sm_count * 16.0) * 1.1 + 2.0;
            const double cost = std::max(lat, thr) + static_cast<double>(std::min(rows_cap, 8)) * K / 2048.0;
            if (!found || cost < best - 1e-9) {
                found = true;
                best = cost;
                tp.p = lp;
                tp.p.M = rows_cap;
                tp.p.N = N;
                tp.p.K = K;
                tp.p.tiles = tiles;
                tp.p.ksplit_log2 = 0;
                tp.p.s_log2 = 0;
                tp.p.tpi = tk::kWarps;
                tp.p.ipg = tiles;
                tp.p.items_q = static_cast<int>(jobs);
                tp.p.items_r = aligned;  // stream-K: 1 = group-aligned CTA ranges
                tp.p.nbox = nbox;
                tp.p.stages = stages;
                tp.p.sstride = sstride;
                tp.nc = nc;
                tp.grid_x = static_cast<int>(units);
                tp.grid_y = 1;
                tp.smem = smem;
                tp.sk = true;
            }
          }
        }
    }
    if (found && cost_out) *cost_out = best;
    return found;
}

// Codes [rows, K/2] as (128 B, K/256, rows) with a 128-byte swizzle, scales [rows, K/16] as
// (16 B, K/256, rows); boxes of NC segments x 16 rows.
bool encode_tile_maps(CUtensorMap* wmap, CUtensorMap* smap, const uint8_t* w, const uint8_t* s, int64_t rows,
                      int K, int nc) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint32_t estr[3] = {1, 1, 1};
    if (wmap) {
        const cuuint64_t dims[3] = {128, static_cast<cuuint64_t>(K / 256), static_cast<cuuint64_t>(rows)};
        const cuuint64_t strides[2] = {128, static_cast<cuuint64_t>(K / 2)};
        const cuuint32_t box[3] = {128, static_cast<cuuint32_t>(nc), 16};
        if (enc(wmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(w), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    if (smap) {
        const cuuint64_t dims[3] = {16, static_cast<cuuint64_t>(K / 256), static_cast<cuuint64_t>(rows)};
        const cuuint64_t strides[2] = {16, static_cast<cuuint64_t>(K / 16)};
        const cuuint32_t box[3] = {16, static_cast<cuuint32_t>(nc), 16};
        if (enc(smap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(s), dims, strides, box, estr,
                CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
            return false;
    }
    return true;
}

// Index plane of dictionary scales viewed as (160 B, K/256, tiles): one record per box segment.
bool encode_sd_map(CUtensorMap* smap, const uint8_t* plane, int64_t tiles, int K, int nc) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint32_t estr[3] = {1, 1, 1};
    const cuuint64_t dims[3] = {static_cast<cuuint64_t>(kSdRecord), static_cast<cuuint64_t>(K / 256),
                                static_cast<cuuint64_t>(tiles)};
    const cuuint64_t strides[2] = {static_cast<cuuint64_t>(kSdRecord), static_cast<cuuint64_t>(K / 256) * kSdRecord};
    const cuuint32_t box[3] = {static_cast<cuuint32_t>(kSdRecord), static_cast<cuuint32_t>(nc), 1};
    return enc(smap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<uint8_t*>(plane), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <int NC, bool MOE, bool SK, bool SWI = false, bool SD = false>
cudaError_t launch_tile_nc(const TilePlan& tp, cudaStream_t st) {
    auto kern = [] {
        if constexpr (SK) return gemv_tile_sk_kernel<NC, MOE, SD>;
        else return gemv_tile_kernel<NC, MOE, SWI, SD>;
    }();
    static bool done[64] = {};
    cudaError_t e = allow_max_smem(kern, done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(tp.grid_x, tp.grid_y);
    cfg.blockDim = dim3(tk::kThreads);
    cfg.dynamicSmemBytes = tp.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    if (tp.p.s_log2 > 0) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = 1u << tp.p.s_log2;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (g_pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, tp.p);
}

// Launch slot of the phase trace: consecutive tile-kernel launches use consecutive slots.
int g_trace_next = 0;

cudaError_t launch_tile(const TilePlan& tp_in, cudaStream_t st, bool moe, bool sd = false) {
    TilePlan tp = tp_in;
    if (NVFP4_PHASE_TRACE) {
        std::lock_guard<std::mutex> lk(g_mu);
        tp.p.trace_slot = g_trace_next;
        g_trace_next = (g_trace_next + 1) % kTraceLaunches;
    }
    if (sd) {
        if (moe) {
            if (!tp.sk) return cudaErrorInvalidValue;
            return tp.nc == 2 ? launch_tile_nc<2, true, true, false, true>(tp, st)
                              : launch_tile_nc<1, true, true, false, true>(tp, st);
        }
        return tp.nc == 2 ? launch_tile_nc<2, false, false, false, true>(tp, st)
                          : launch_tile_nc<1, false, false, false, true>(tp, st);
    }
    if (moe && tp.sk) return tp.nc == 2 ? launch_tile_nc<2, true, true>(tp, st) : launch_tile_nc<1, true, true>(tp, st);
    if (moe) return tp.nc == 2 ? launch_tile_nc<2, true, false>(tp, st) : launch_tile_nc<1, true, false>(tp, st);
    if (tp.p.swiglu)
        return tp.nc == 2 ? launch_tile_nc<2, false, false, true>(tp, st) : launch_tile_nc<1, false, false, true>(tp, st);
    return tp.nc == 2 ? launch_tile_nc<2, false, false>(tp, st) : launch_tile_nc<1, false, false>(tp, st);
}

cudaError_t launch_simple(const SimpleParams& sp, int64_t cols, cudaStream_t st) {
    const int per_block = kSimpleThreads / 32;
    const int64_t blocks = (cols + per_block - 1) / per_block;
    if (blocks > 0x7fffffff) return cudaErrorInvalidValue;
    const dim3 grid(static_cast<unsigned>(blocks)), block(kSimpleThreads);
    const int mt = sp.moe ? 1 : sp.M;
    switch (mt) {
        case 1: gemv_simple_kernel<1><<<grid, block, 0, st>>>(sp); break;
        case 2: gemv_simple_kernel<2><<<grid, block, 0, st>>>(sp); break;
        case 3: gemv_simple_kernel<3><<<grid, block, 0, st>>>(sp); break;
        case 4: gemv_simple_kernel<4><<<grid, block, 0, st>>>(sp); break;
        case 5: gemv_simple_kernel<5><<<grid, block, 0, st>>>(sp); break;
        case 6: gemv_simple_kernel<6><<<grid, block, 0, st>>>(sp); break;
        case 7: gemv_simple_kernel<7><<<grid, block, 0, st>>>(sp); break;
        case 8: gemv_simple_kernel<8><<<grid, block, 0, st>>>(sp); break;
        default: return cudaErrorInvalidValue;
    }
    return cudaGetLastError();
}

nvfp4_status check_out(int y_type) {
    return (y_type == NVFP4_OUT_F32 || y_type == NVFP4_OUT_BF16) ? NVFP4_OK : NVFP4_ERR_DTYPE;
}

nvfp4_status zero_output(void* y, int64_t elems, int y_type, cudaStream_t st) {
    const size_t bytes = static_cast<size_t>(elems) * (y_type == NVFP4_OUT_BF16 ? 2 : 4);
    const cudaError_t e = cudaMemsetAsync(y, 0, bytes, st);
    return e == cudaSuccess ? NVFP4_OK : cuda_fail(e);
}

// Tile-kernel plans with their encoded tensor maps, reused by later calls with the same device,
// shape, kernel selection and weight pointers (a tensor map holds nothing else: the same
// pointer and shape always give the same map). Direct-mapped; a colliding call replaces the
// entry. Per-call values (x, y, scales, output type) are filled in after the lookup.
struct PlanKey {
    int dev, kind, M, N, K, groups, variant, E, T, top_k, xps;
    const void* w[2];
    const void* s[2];
    bool operator==(const PlanKey& o) const { return std::memcmp(this, &o, sizeof(PlanKey)) == 0; }
};
struct PlanEntry {
    PlanKey key;
    bool used;
    bool tile;       // false: the tile kernel does not take this call
    TilePlan tp;
};
constexpr int kPlanCacheSize = 64;
PlanEntry g_plan_cache[kPlanCacheSize];

PlanKey make_key(int dev, int kind, int M, int N, int K, int groups, const uint8_t* const* w,
                 const uint8_t* const* s, int E = 0, int T = 0, int top_k = 0, int xps = 0) {
    PlanKey k;
    std::memset(&k, 0, sizeof k);  // padding included: keys compare as bytes
    k.dev = dev; k.kind = kind; k.M = M; k.N = N; k.K = K; k.groups = groups; k.variant = g_variant;
    k.E = E; k.T = T; k.top_k = top_k; k.xps = xps;
    for (int i = 0; i < 2; ++i) {
        k.w[i] = w[i < groups ? i : 0];
        k.s[i] = s[i < groups ? i : 0];
    }
    return k;
}

uint32_t key_slot(const PlanKey& k) {
    const unsigned char* b = reinterpret_cast<const unsigned char*>(&k);
    uint32_t h = 2166136261u;  // FNV-1a over the key's bytes
    for (size_t i = 0; i < sizeof k; ++i) h = (h ^ b[i]) * 16777619u;
    return h % kPlanCacheSize;
}

// The cached tile plan for key k, built by `make` (returns false when the tile kernel does not
// take the call) on a miss. Returns whether the tile kernel takes the call; *out gets the plan.
template <typename F>
bool cached_tile_plan(const PlanKey& k, TilePlan* out, F&& make) {
    const uint32_t slot = key_slot(k);
    {
        std::lock_guard<std::mutex> lk(g_mu);
        const PlanEntry& e = g_plan_cache[slot];
        if (e.used && e.key == k) {
            if (e.tile) *out = e.tp;
            return e.tile;
        }
    }
    TilePlan tp{};
    const bool tile = make(tp);
    std::lock_guard<std::mutex> lk(g_mu);
    PlanEntry& e = g_plan_cache[slot];
    e.key = k;
    e.used = true;
    e.tile = tile;
    e.tp = tp;
    if (tile) *out = tp;
    return tile;
}

// Dense (groups = 1) and gate/up (groups = 2) calls; swiglu: gate/up with the fused
// activation, y [M, N] = silu(clamp(gate)) * clamp(up).
nvfp4_status run_dense(const uint8_t* const* w, const uint8_t* const* s, const float* g, int groups,
                       const uint16_t* x, void* y, int y_type, int M, int N, int K, cudaStream_t st,
                       bool swiglu = false, float clamp = 0.f) {
    if (!x || !y) return NVFP4_ERR_NULL;
    for (int i = 0; i < groups; ++i)
        if (!w[i] || !s[i]) return NVFP4_ERR_NULL;
    if (M < 0 || N < 0 || K < 0 || M > 8 || K % 16 != 0) return NVFP4_ERR_SHAPE;
    const nvfp4_status so = check_out(y_type);
    if (so != NVFP4_OK) return so;
    if (M == 0 || N == 0) return NVFP4_OK;
    const int64_t ldy = swiglu ? N : static_cast<int64_t>(groups) * N;  // output columns
    if (K == 0) return zero_output(y, static_cast<int64_t>(M) * ldy, y_type, st);  // silu(0) * 0 = 0
    int dev = 0;
    const DeviceInfo* d = device_info(&dev);
    if (!d) return cuda_fail(cudaGetLastError());
    TilePlan tpl{};
    const bool x_ok = (reinterpret_cast<uintptr_t>(x) & 15) == 0;  // the only x property a plan reads
    const PlanKey key = make_key(dev, (swiglu ? 4 : groups) + (x_ok ? 0 : 8), M, N, K, groups, w, s);
    const bool tile = cached_tile_plan(key, &tpl, [&](TilePlan& tp) {
        if (!plan_tile(tp, M, N, K, groups, *d, w, s, x, false, 0, 0, swiglu)) return false;
        for (int i = 0; i < groups; ++i)
            if (!encode_tile_maps(&tp.p.wmap[i], &tp.p.smap[i], w[i], s[i], N, K, tp.nc)) return false;
        if (groups == 1) {
            tp.p.wmap[1] = tp.p.wmap[0];
            tp.p.smap[1] = tp.p.smap[0];
        }
        return true;
    });
    if (tile) {
        TileParams& p = tpl.p;
        p.x = x;
        p.y = y;
        p.g[0] = g[0];
        p.g[1] = g[groups > 1 ? 1 : 0];
        p.ldy = ldy;
        p.swiglu = swiglu ? 1 : 0;
        p.clamp = clamp;
        p.out_bf16 = y_type == NVFP4_OUT_BF16;
        p.force_f32 = g_variant == 2;
        p.wait_ns = g_wait_ns;
        const cudaError_t e = launch_tile(tpl, st, false);
        if (e != cudaSuccess) return cuda_fail(e);
        const cudaError_t e2 = cudaGetLastError();
        return e2 == cudaSuccess ? NVFP4_OK : cuda_fail(e2);
    }
    Plan pl{};
    if (!swiglu && plan_dense(pl, M, N, K, groups, *d, w, s, x)) {
        Params& p = pl.p;
        for (int i = 0; i < 2; ++i) {
            p.w[i] = w[i < groups ? i : 0];
            p.s[i] = s[i < groups ? i : 0];
            p.g[i] = g[i < groups ? i : 0];
        }
        p.x = x;
        p.y = y;
        p.ldy = static_cast<int64_t>(groups) * N;
        p.out_bf16 = y_type == NVFP4_OUT_BF16;
        p.wait_ns = g_wait_ns;
        p.force_f32 = g_variant == 2;
        const cudaError_t e = dispatch_stream(pl, st);
        if (e != cudaSuccess) return cuda_fail(e);
        const cudaError_t e2 = cudaGetLastError();
        return e2 == cudaSuccess ? NVFP4_OK : cuda_fail(e2);
    }
    SimpleParams sp{};
    for (int i = 0; i < 2; ++i) {
        sp.w[i] = w[i < groups ? i : 0];
        sp.s[i] = s[i < groups ? i : 0];
        sp.g[i] = g[i < groups ? i : 0];
    }
    sp.x = x; sp.y = y; sp.ldy = ldy; sp.out_bf16 = y_type == NVFP4_OUT_BF16;
    sp.M = M; sp.N = N; sp.K = K; sp.groups = groups;
    sp.swiglu = swiglu ? 1 : 0;
    sp.clamp = clamp;
    const cudaError_t e = launch_simple(sp, ldy, st);
    return e == cudaSuccess ? NVFP4_OK : cuda_fail(e);
}

// Dense GEMV with dictionary scales: the tile kernel's SD form, else the byte-load kernel.
nvfp4_status run_sdict_dense(const uint8_t* w, const uint8_t* plane, const uint8_t* dict, float g, const uint16_t* x,
                             void* y, int y_type, int M, int N, int K, cudaStream_t st) {
    if (!w || !plane || !dict || !x || !y) return NVFP4_ERR_NULL;
    if (M < 0 || N < 0 || K < 0 || M > 8 || K % 256 != 0) return NVFP4_ERR_SHAPE;
    const nvfp4_status so = check_out(y_type);
    if (so != NVFP4_OK) return so;
    if (M == 0 || N == 0) return NVFP4_OK;
    if (K == 0) return zero_output(y, static_cast<int64_t>(M) * N, y_type, st);
    int dev = 0;
    const DeviceInfo* d = device_info(&dev);
    if (!d) return cuda_fail(cudaGetLastError());
    const uint8_t* wv[1] = {w};
    const uint8_t* sv[1] = {plane};
    const bool x_ok = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    TilePlan tpl{};
    const PlanKey key = make_key(dev, 16 + (x_ok ? 0 : 8), M, N, K, 1, wv, sv);
    const bool tile = cached_tile_plan(key, &tpl, [&](TilePlan& tp) {
        if (!plan_tile(tp, M, N, K, 1, *d, wv, sv, x, false, 0, 0, false, true, true)) return false;
        if (!encode_tile_maps(&tp.p.wmap[0], nullptr, w, nullptr, N, K, tp.nc)) return false;
        if (!encode_sd_map(&tp.p.smap[0], plane, (N + 15) / 16, K, tp.nc)) return false;
        tp.p.wmap[1] = tp.p.wmap[0];
        tp.p.smap[1] = tp.p.smap[0];
        return true;
    });
    if (tile) {
        TileParams& p = tpl.p;
        p.x = x;
        p.y = y;
        p.g[0] = p.g[1] = g;
        p.ldy = N;
        p.out_bf16 = y_type == NVFP4_OUT_BF16;
        p.force_f32 = g_variant == 2;
        p.wait_ns = g_wait_ns;
        p.sd_dict = dict;
        const cudaError_t e = launch_tile(tpl, st, false, true);
        if (e != cudaSuccess) return cuda_fail(e);
        const cudaError_t e2 = cudaGetLastError();
        return e2 == cudaSuccess ? NVFP4_OK : cuda_fail(e2);
    }
    SimpleParams sp{};
    sp.w[0] = sp.w[1] = w;
    sp.s[0] = sp.s[1] = plane;
    sp.g[0] = sp.g[1] = g;
    sp.x = x; sp.y = y; sp.ldy = N; sp.out_bf16 = y_type == NVFP4_OUT_BF16;
    sp.M = M; sp.N = N; sp.K = K; sp.groups = 1;
    sp.sd = 1;
    sp.sd_dict = dict;
    const cudaError_t e = launch_simple(sp, N, st);
    return e == cudaSuccess ? NVFP4_OK : cuda_fail(e);
}

// Routed-expert GEMV with dictionary scales: the stream-K tile kernel's SD form with
// group-aligned ranges for up to 32 slots, else the byte-load kernel.
nvfp4_status run_sdict_moe(const uint8_t* w, const uint8_t* plane, const uint8_t* dict, const float* gs, int E,
                           const int32_t* ids, int T, int top_k, const uint16_t* x, int x_per_slot, void* y,
                           int y_type, int N, int K, int32_t* status_dev, cudaStream_t st) {
    if (!w || !plane || !dict || !gs || !ids || !x || !y) return NVFP4_ERR_NULL;
    if (E < 1 || T < 0 || top_k < 0 || N < 0 || K < 0 || K % 256 != 0) return NVFP4_ERR_SHAPE;
    if (static_cast<int64_t>(T) * top_k > (1 << 24)) return NVFP4_ERR_UNSUPPORTED;
    const nvfp4_status so = check_out(y_type);
    if (so != NVFP4_OK) return so;
    const int slots = T * top_k;
    if (slots == 0 || N == 0) return NVFP4_OK;
    if (K == 0) return zero_output(y, static_cast<int64_t>(slots) * N, y_type, st);
    int dev = 0;
    const DeviceInfo* d = device_info(&dev);
    if (!d) return cuda_fail(cudaGetLastError());
    const int64_t tiles_n = (N + 15) / 16;
    if (slots <= kMaxMoeSlots && static_cast<int64_t>(E) * N <= (1 << 30)) {
        TilePlan tpl{};
        const uint8_t* wv[1] = {w};
        const uint8_t* sv[1] = {plane};
        const int xrows = x_per_slot ? slots : T;
        const bool x_ok = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
        const PlanKey key = make_key(dev, 17 + (x_ok ? 0 : 8), 8, N, K, 1, wv, sv, E, T, top_k, x_per_slot ? 1 : 0);
        const bool tile = cached_tile_plan(key, &tpl, [&](TilePlan& tp) {
            if (!plan_tile(tp, 8, N, K, expected_groups(E, T, top_k), *d, wv, sv, x, true, xrows, slots, false, true,
                           true))
                return false;
            if (!tp.sk || !tp.p.items_r) return false;  // group-aligned stream-K only
            if (!encode_tile_maps(&tp.p.wmap[0], nullptr, w, nullptr, static_cast<int64_t>(E) * N, K, tp.nc))
                return false;
            if (!encode_sd_map(&tp.p.smap[0], plane, static_cast<int64_t>(E) * tiles_n, K, tp.nc)) return false;
            tp.p.wmap[1] = tp.p.wmap[0];
            tp.p.smap[1] = tp.p.smap[0];
            return true;
        });
        if (tile) {
            TileParams& p = tpl.p;
            p.x = x;
            p.y = y;
            p.ldy = N;
            p.out_bf16 = y_type == NVFP4_OUT_BF16;
            p.force_f32 = g_variant == 2;
            p.wait_ns = g_wait_ns;
            p.ids = ids;
            p.g_dev = gs;
            p.status_user = status_dev;
            p.E = E;
            p.top_k = top_k;
            p.slots = slots;
            p.x_per_slot = x_per_slot ? 1 : 0;
            p.sd_dict = dict;
            p.sd_tiles = static_cast<int>(tiles_n);
            const cudaError_t e = launch_tile(tpl, st, true, true);
            if (e != cudaSuccess) return cuda_fail(e);
            const cudaError_t e2 = cudaGetLastError();
            return e2 == cudaSuccess ? NVFP4_OK : cuda_fail(e2);
        }
    }
    SimpleParams sp{};
    sp.w[0] = sp.w[1] = w;
    sp.s[0] = sp.s[1] = plane;
    sp.g_dev = gs;
    sp.ids = ids;
    sp.status_user = status_dev;
    sp.x = x; sp.y = y; sp.ldy = N; sp.out_bf16 = y_type == NVFP4_OUT_BF16;
    sp.M = 1; sp.N = N; sp.K = K; sp.groups = 1;
    sp.moe = 1; sp.E = E; sp.top_k = top_k; sp.x_per_slot = x_per_slot ? 1 : 0; sp.slots = slots;
    sp.sd = 1;
    sp.sd_dict = dict;
    const cudaError_t e = launch_simple(sp, static_cast<int64_t>(slots) * N, st);
    return e == cudaSuccess ? NVFP4_OK : cuda_fail(e);
}

// ------------------------------------------------------------------ the FFN block (host)

// Bytes of the FFN workspace: the counters' lines (kFfnSyncBytes: the finished-CTA count, then
// one counter per phase-B K slice, each in its own 128-byte line), then h as bf16 [M, I] (rows of
// 2 I bytes, back to back), rounded up to 256 bytes.
int64_t ffn_workspace_bytes(int M, int I) {
    return kFfnSyncBytes + (static_cast<int64_t>(M) * I * 2 + 255) / 256 * 256;
}

struct FfnPlan {
    FfnParams p;
    int nc;
    int grid;
    uint32_t smem;
};

// Cost of one phase in units of a warp's 128-element step, as plan_tile prices a per-item
// plan on `units` CTAs: the larger of the latency term (items of the busiest CTA, each with its
// steps and reduction) and the throughput term, plus the staging of x.
double ffn_phase_cost(long long items, int ksplit, int nc, int nbmax, int M, int K, long long units, int sms) {
    const long long ipu = (items + units - 1) / units;
    const double spw = 2.0 * nc * nbmax;
    const double lat = static_cast<double>(ipu) * (spw + (ksplit > 1 ? 2.0 : 0.3));
    const double thr = static_cast<double>(items) * tk::kWarps * spw / (sms * 16.0) * 1.1;
    return std::max(lat, thr) + static_cast<double>(M) * K / 2048.0;
}

// One-launch plan for the FFN block: phase A (gate/up + SwiGLU, K = H, I outputs) and phase B
// (down, K = I, H outputs) on 2 CTAs per SM, one ring for both, and x/h staging that fits beside
// it. The x region holds the larger of A's x slices plus its pair buffer (cpart) and B's h
// slices: a CTA's warps are past its last A item's barrier, so done with both, before any of them
// stages h. False when the block's weights exceed kFfnFusedMaxBytes or no such plan fits.
bool plan_ffn(FfnPlan& fp, int M, int H, int I, const DeviceInfo& d) {
    if (g_variant == 1 || g_variant == 3) return false;
    if (M < 1 || M > 8 || H <= 0 || I <= 0 || H % 256 || I % 256 || H > (1 << 27) || I > (1 << 27)) return false;
    // each phase priced as the separate launch would be: a fused plan whose phase costs far
    // more (a decomposition squeezed to fit beside the other phase's x) is not taken
    const uint8_t* fake = reinterpret_cast<const uint8_t*>(static_cast<uintptr_t>(256));
    const uint8_t* fw[2] = {fake, fake};
    double solo_a = 0.0, solo_b = 0.0;
    TilePlan solo{};
    if (!plan_tile(solo, M, I, H, 2, d, fw, fw, fake, false, 0, 0, true, false, false, &solo_a) ||
        !plan_tile(solo, M, H, I, 1, d, fw, fw, fake, false, 0, 0, false, false, false, &solo_b))
        return false;
    const long long units = static_cast<long long>(d.sm_count) * 2;
    const uint32_t limit = static_cast<uint32_t>(d.smem_per_sm / 2 - 1024);
    bool found = false;
    double best = 0.0;
    // one launch only for latency-bound blocks: measured, the shared expert (H = 4096, I = 768,
    // M = 2, 5.3 MB) ran 10.7 us a step in one launch and 10.8 in two, while the 12288-wide FFN
    // (85 MB) ran 26.5 to 27.8 in one and 23.2 in two
    if (3.0 * H * I * 9.0 / 16.0 > static_cast<double>(kFfnFusedMaxBytes)) return false;
    for (int nc = 2; nc >= 1; --nc) {
        if ((H / 256) % nc || (I / 256) % nc) continue;
        if (NVFP4_TILE_NC && nc != NVFP4_TILE_NC) continue;
        const int nbox_a = H / 256 / nc, nbox_b = I / 256 / nc;
        const int tiles_a = 2 * ((I + 15) / 16), tiles_b = (H + 15) / 16;
        for (int la = 0; la <= 2; ++la) {       // A: tpi >= 2 (whole gate/up pairs)
            const int ka = 1 << la;
            if (ka > nbox_a) break;
            const int tpi_a = tk::kWarps / ka;
            const long long items_a = (tiles_a + tpi_a - 1) / tpi_a;
            const int nbmax_a = (nbox_a + ka - 1) / ka;
            const uint32_t sstride_a = static_cast<uint32_t>(nbmax_a) * nc * 512u + 64u;
            const uint32_t xa = align_up(static_cast<uint32_t>(ka * M) * sstride_a, 128);
            for (int lb = 0; lb <= 3; ++lb) {
                const int kb = 1 << lb;
                if (kb > nbox_b) break;
                const int tpi_b = tk::kWarps / kb;
                const long long items_b = (tiles_b + tpi_b - 1) / tpi_b;
                const int nbmax_b = (nbox_b + kb - 1) / kb;
                const uint32_t sstride_b = static_cast<uint32_t>(nbmax_b) * nc * 512u + 64u;
                const uint32_t xb = align_up(static_cast<uint32_t>(kb * M) * sstride_b, 128);
                const uint32_t cpart = 2u * tk::kWarps * 16 * 8 * 4u;
                const uint32_t xreg = std::max(xa + cpart, xb);
                const uint32_t red = (ka > 1 || kb > 1) ? 2u * tk::kRedFloats * 4u : 0u;
                for (int st = tk::kMaxStages; st >= 2; --st) {
                    TileParams q{};
                    uint32_t off = 0;
                    q.ring_w = off;
                    off += static_cast<uint32_t>(tk::kWarps * st * nc) * 2048u;
                    q.ring_s = off;
                    off += static_cast<uint32_t>(tk::kWarps * st * nc) * 256u;
                    q.x_off = off;
                    q.cpart_off = off + xa;
                    off += xreg;
                    q.red_off = off;
                    off += red;
                    q.misc_off = off;
                    off += align_up(tk::kWarps * 32 + tk::kWarps * 32 * 4, 128);
                    q.bar_off = off;
                    off += tk::kWarps * tk::kMaxStages * 8;
                    q.moe_off = q.sdtab_off = off;
                    const uint32_t total = off + 1024;
                    if (total > limit) continue;
                    const double ca = ffn_phase_cost(items_a, ka, nc, nbmax_a, M, H, units, d.sm_count);
                    const double cb = ffn_phase_cost(items_b, kb, nc, nbmax_b, M, I, units, d.sm_count);
                    const double cost = ca + cb;
                    if (ca > 1.5 * solo_a || cb > 1.5 * solo_b) break;
                    if (!found || cost < best - 1e-9) {
                        found = true;
                        best = cost;
                        TileParams a = q, b = q;
                        a.M = b.M = M;
                        a.N = I; a.K = H; a.tiles = tiles_a; a.ksplit_log2 = la; a.tpi = tpi_a;
                        a.ipg = static_cast<int>(items_a);
                        a.items_q = static_cast<int>(items_a / units);
                        a.items_r = static_cast<int>(items_a % units);
                        a.nbox = nbox_a; a.sstride = sstride_a; a.swiglu = 1;
                        b.N = H; b.K = I; b.tiles = tiles_b; b.ksplit_log2 = lb; b.tpi = tpi_b;
                        b.ipg = static_cast<int>(items_b);
                        b.items_q = static_cast<int>(items_b / units);
                        b.items_r = static_cast<int>(items_b % units);
                        b.nbox = nbox_b; b.sstride = sstride_b;
                        a.stages = b.stages = st;
                        fp.p.a = a;
                        fp.p.b = b;
                        fp.nc = nc;
                        fp.grid = static_cast<int>(units);
                        fp.smem = total;
                    }
                    break;  // the deepest ring that fits
                }
            }
        }
    }
    return found;
}

template <int NC>
cudaError_t launch_ffn_nc(const FfnPlan& fp, cudaStream_t st) {
    auto kern = gemv_ffn_kernel<NC>;
    static bool done[64] = {};
    cudaError_t e = allow_max_smem(kern, done);
    if (e != cudaSuccess) return e;
    cudaLaunchConfig_t cfg{};
    cfg.gridDim = dim3(fp.grid);
    cfg.blockDim = dim3(kFfnThreads);
    cfg.dynamicSmemBytes = fp.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    int na = 0;
    if (g_pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, fp.p);
}

// Whether the fused kernel keeps two CTAs per SM resident at this shared-memory size (the grid
// barrier needs every CTA of the launch resident at once).
template <int NC>
bool ffn_two_per_sm(uint32_t smem) {
    static bool done[64] = {};
    if (allow_max_smem(gemv_ffn_kernel<NC>, done) != cudaSuccess) return false;
    int n = 0;
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, gemv_ffn_kernel<NC>, kFfnThreads, smem) != cudaSuccess) {
        cudaGetLastError();
        return false;
    }
    return n >= 2;
}

struct FfnKey {
    int dev, M, H, I, variant;
    const void* w[3];
    const void* s[3];
    bool operator==(const FfnKey& o) const { return std::memcmp(this, &o, sizeof(FfnKey)) == 0; }
};
struct FfnEntry {
    FfnKey key;
    bool used;
    bool fused;
    FfnPlan fp;
};
constexpr int kFfnCacheSize = 16;
FfnEntry g_ffn_cache[kFfnCacheSize];

// The FFN block: one fused launch when a plan fits with every CTA resident (2 per SM), else the
// gate/up + SwiGLU launch writing h into the workspace, then the down launch reading it.
nvfp4_status run_ffn(const uint8_t* const* w, const uint8_t* const* s, const float* g, const uint16_t* x,
                     float clamp, void* workspace, void* y, int y_type, int M, int H, int I, cudaStream_t st) {
    if (!x || !y || !workspace) return NVFP4_ERR_NULL;
    for (int i = 0; i < 3; ++i)
        if (!w[i] || !s[i]) return NVFP4_ERR_NULL;
    if (!(clamp > 0.f)) return NVFP4_ERR_SHAPE;  // also rejects NaN
    if (M < 0 || H < 0 || I < 0 || M > 8 || H % 16 != 0 || I % 16 != 0) return NVFP4_ERR_SHAPE;
    if (reinterpret_cast<uintptr_t>(workspace) & 255) return NVFP4_ERR_ALIGN;
    const nvfp4_status so = check_out(y_type);
    if (so != NVFP4_OK) return so;
    if (M == 0 || H == 0) return NVFP4_OK;
    if (I == 0) return zero_output(y, static_cast<int64_t>(M) * H, y_type, st);  // an empty down sum
    int dev = 0;
    const DeviceInfo* d = device_info(&dev);
    if (!d) return cuda_fail(cudaGetLastError());
    uint16_t* h = reinterpret_cast<uint16_t*>(static_cast<uint8_t*>(workspace) + kFfnSyncBytes);
    FfnKey key;
    std::memset(&key, 0, sizeof key);
    key.dev = dev; key.M = M; key.H = H; key.I = I; key.variant = g_variant;
    for (int i = 0; i < 3; ++i) {
        key.w[i] = w[i];
        key.s[i] = s[i];
    }
    const bool x_ok = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
    bool w_ok = true;
    for (int i = 0; i < 3; ++i)
        w_ok = w_ok && !(reinterpret_cast<uintptr_t>(w[i]) & 15) && !(reinterpret_cast<uintptr_t>(s[i]) & 15);
    FfnPlan fp{};
    bool fused = false;
    if (x_ok && w_ok) {
        uint32_t slot = 2166136261u;
        const unsigned char* kb = reinterpret_cast<const unsigned char*>(&key);
        for (size_t i = 0; i < sizeof key; ++i) slot = (slot ^ kb[i]) * 16777619u;
        slot %= kFfnCacheSize;
        bool hit = false;
        {
            std::lock_guard<std::mutex> lk(g_mu);
            const FfnEntry& e = g_ffn_cache[slot];
            if (e.used && e.key == key) {
                hit = true;
                fused = e.fused;
                if (fused) fp = e.fp;
            }
        }
        if (!hit) {
            fused = tensor_map_encoder() && plan_ffn(fp, M, H, I, *d);
            if (fused) fused = fp.nc == 2 ? ffn_two_per_sm<2>(fp.smem) : ffn_two_per_sm<1>(fp.smem);
            if (fused) {
                fused = encode_tile_maps(&fp.p.a.wmap[0], &fp.p.a.smap[0], w[0], s[0], I, H, fp.nc) &&
                        encode_tile_maps(&fp.p.a.wmap[1], &fp.p.a.smap[1], w[1], s[1], I, H, fp.nc) &&
                        encode_tile_maps(&fp.p.b.wmap[0], &fp.p.b.smap[0], w[2], s[2], H, I, fp.nc);
                fp.p.b.wmap[1] = fp.p.b.wmap[0];
                fp.p.b.smap[1] = fp.p.b.smap[0];
            }
            std::lock_guard<std::mutex> lk(g_mu);
            FfnEntry& e = g_ffn_cache[slot];
            e.key = key;
            e.used = true;
            e.fused = fused;
            e.fp = fp;
        }
    }
    if (fused) {
        TileParams& a = fp.p.a;
        TileParams& b = fp.p.b;
        a.x = x;
        a.y = h;
        a.g[0] = g[0];
        a.g[1] = g[1];
        a.ldy = I;
        a.clamp = clamp;
        a.out_bf16 = 1;
        b.x = h;
        b.y = y;
        b.g[0] = b.g[1] = g[2];
        b.ldy = H;
        b.out_bf16 = y_type == NVFP4_OUT_BF16;
        a.force_f32 = b.force_f32 = g_variant == 2;
        a.wait_ns = b.wait_ns = g_wait_ns;
        fp.p.sync = static_cast<uint32_t*>(workspace);
        if (NVFP4_PHASE_TRACE) {
            std::lock_guard<std::mutex> lk(g_mu);
            a.trace_slot = g_trace_next;
            g_trace_next = (g_trace_next + 1) % kTraceLaunches;
        }
        const cudaError_t e = fp.nc == 2 ? launch_ffn_nc<2>(fp, st) : launch_ffn_nc<1>(fp, st);
        if (e != cudaSuccess) return cuda_fail(e);
        const cudaError_t e2 = cudaGetLastError();
        return e2 == cudaSuccess ? NVFP4_OK : cuda_fail(e2);
    }
    const uint8_t* wgu[2] = {w[0], w[1]};
    const uint8_t* sgu[2] = {s[0], s[1]};
    const float ggu[2] = {g[0], g[1]};
    nvfp4_status r = run_dense(wgu, sgu, ggu, 2, x, h, NVFP4_OUT_BF16, M, I, H, st, true, clamp);
    if (r != NVFP4_OK) return r;
    const uint8_t* wd[1] = {w[2]};
    const uint8_t* sd[1] = {s[2]};
    const float gd[1] = {g[2]};
    return run_dense(wd, sd, gd, 1, h, y, y_type, M, H, I, st);
}

// ------------------------------------------------------------------ the FFN block without a caller workspace

// The FFN block's workspace as a file-scope device array, for callers that cannot hand the
// library a workspace: a C caller with no device allocator of its own, or one whose allocator
// must not run on its decode path. 256 KB holds the counters and h up to M * I = 130048 (M = 8 at
// I = 12288). One array per device and process: calls that overlap in time (other streams, other
// host threads without ordering) share it and corrupt each other's h and counters.
constexpr int64_t kFfnStaticScratchBytes = 256ll << 10;
static __device__ __align__(256) uint8_t g_ffn_scratch[kFfnStaticScratchBytes];

// The array's device address on the current device, looked up once per device; the first lookup
// also zeroes the counters on `st` (the array is zero at load; this makes it explicit).
void* ffn_static_scratch(int dev, cudaStream_t st) {
    static void* addr[64] = {};
    std::lock_guard<std::mutex> lk(g_mu);
    if (dev < 0 || dev >= 64) return nullptr;
    if (!addr[dev]) {
        void* a = nullptr;
        if (cudaGetSymbolAddress(&a, g_ffn_scratch) != cudaSuccess) return nullptr;
        if (cudaMemsetAsync(a, 0, kFfnSyncBytes, st) != cudaSuccess) return nullptr;
        addr[dev] = a;
    }
    return addr[dev];
}

}  // namespace nvfp4

using namespace nvfp4;

extern "C" {

nvfp4_status nvfp4_gemv_sdict(const uint8_t* w_packed, const uint8_t* scale_idx, const uint8_t* scale_dict,
                              float global_scale, const uint16_t* x, void* y, nvfp4_out_t y_type, int M, int N,
                              int K, void* stream) {
    return run_sdict_dense(w_packed, scale_idx, scale_dict, global_scale, x, y, y_type, M, N, K,
                           static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_moe_gemv_sdict(const uint8_t* w_packed, const uint8_t* scale_idx, const uint8_t* scale_dict,
                                  const float* global_scales, int E, const int32_t* expert_ids, int T, int top_k,
                                  const uint16_t* x, int x_per_slot, void* y, nvfp4_out_t y_type, int N, int K,
                                  int32_t* status_dev, void* stream) {
    return run_sdict_moe(w_packed, scale_idx, scale_dict, global_scales, E, expert_ids, T, top_k, x, x_per_slot, y,
                         y_type, N, K, status_dev, static_cast<cudaStream_t>(stream));
}

int64_t nvfp4_sdict_plane_bytes(int N, int K) {
    if (N < 0 || K < 0 || K % 256 != 0) return -1;
    return sd_plane_bytes(N, K);
}

int nvfp4_sdict_encode(const uint8_t* scales, int N, int K, uint8_t* plane_out, uint8_t* dict_out) {
    if (!dict_out || N < 0 || K < 0 || K % 256 != 0 || (N > 0 && K > 0 && (!scales || !plane_out))) return -2;
    const int64_t blocks = static_cast<int64_t>(K) / 16;
    bool used[256] = {};
    for (int64_t i = 0; i < static_cast<int64_t>(N) * blocks; ++i) used[scales[i]] = true;
    int index_of[256];
    int count = 0;
    uint8_t table[32] = {};
    for (int c = 0; c < 256; ++c) {
        if (!used[c]) continue;
        if (count == 32) return -1;  // more than 32 codes: the tensor stays plain
        index_of[c] = count;
        table[count++] = static_cast<uint8_t>(c);
    }
    for (int i = count; i < 32; ++i) table[i] = count ? table[count - 1] : 0;
    std::memcpy(dict_out, table, 32);
    if (sd_plane_bytes(N, K) > 0) std::memset(plane_out, 0, static_cast<size_t>(sd_plane_bytes(N, K)));
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < blocks; ++b) {
            const uint32_t v = static_cast<uint32_t>(index_of[scales[n * blocks + b]]);
            uint8_t* rec = plane_out + ((n >> 4) * (K >> 8) + (b >> 4)) * kSdRecord;
            const uint32_t bit = static_cast<uint32_t>(((n & 15) * 16 + (b & 15)) * 5);
            for (int i = 0; i < 5; ++i)
                if ((v >> i) & 1u) rec[(bit + i) >> 3] |= static_cast<uint8_t>(1u << ((bit + i) & 7));
        }
    }
    return count;
}

nvfp4_status nvfp4_gemv(const uint8_t* w_packed, const uint8_t* w_scales, float global_scale,
                        const uint16_t* x, void* y, nvfp4_out_t y_type, int M, int N, int K, void* stream) {
    const uint8_t* w[1] = {w_packed};
    const uint8_t* s[1] = {w_scales};
    const float g[1] = {global_scale};
    return run_dense(w, s, g, 1, x, y, y_type, M, N, K, static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_gemv_gate_up(const uint8_t* w_gate, const uint8_t* s_gate, float g_gate,
                                const uint8_t* w_up, const uint8_t* s_up, float g_up,
                                const uint16_t* x, void* y, nvfp4_out_t y_type,
                                int M, int N, int K, void* stream) {
    const uint8_t* w[2] = {w_gate, w_up};
    const uint8_t* s[2] = {s_gate, s_up};
    const float g[2] = {g_gate, g_up};
    return run_dense(w, s, g, 2, x, y, y_type, M, N, K, static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_gemv_gate_up_swiglu(const uint8_t* w_gate, const uint8_t* s_gate, float g_gate,
                                       const uint8_t* w_up, const uint8_t* s_up, float g_up,
                                       const uint16_t* x, float clamp_limit, void* y, nvfp4_out_t y_type,
                                       int M, int N, int K, void* stream) {
    if (!(clamp_limit > 0.f)) return NVFP4_ERR_SHAPE;  // also rejects NaN
    const uint8_t* w[2] = {w_gate, w_up};
    const uint8_t* s[2] = {s_gate, s_up};
    const float g[2] = {g_gate, g_up};
    return run_dense(w, s, g, 2, x, y, y_type, M, N, K, static_cast<cudaStream_t>(stream), true, clamp_limit);
}

int64_t nvfp4_ffn_workspace_bytes(int M, int I) {
    if (M < 0 || M > 8 || I < 0) return -1;
    return ffn_workspace_bytes(M, I);
}

nvfp4_status nvfp4_ffn_swiglu(const uint8_t* w_gate, const uint8_t* s_gate, float g_gate,
                              const uint8_t* w_up, const uint8_t* s_up, float g_up,
                              const uint8_t* w_down, const uint8_t* s_down, float g_down,
                              const uint16_t* x, float clamp_limit, void* workspace,
                              void* y, nvfp4_out_t y_type, int M, int H, int I, void* stream) {
    const uint8_t* w[3] = {w_gate, w_up, w_down};
    const uint8_t* s[3] = {s_gate, s_up, s_down};
    const float g[3] = {g_gate, g_up, g_down};
    return run_ffn(w, s, g, x, clamp_limit, workspace, y, y_type, M, H, I, static_cast<cudaStream_t>(stream));
}

nvfp4_status nvfp4_ffn_swiglu_static(const uint8_t* w_gate, const uint8_t* s_gate, float g_gate,
                                     const uint8_t* w_up, const uint8_t* s_up, float g_up,
                                     const uint8_t* w_down, const uint8_t* s_down, float g_down,
                                     const uint16_t* x, float clamp_limit, void* y, nvfp4_out_t y_type,
                                     int M, int H, int I, void* stream) {
    if (M < 0 || M > 8 || I < 0) return NVFP4_ERR_SHAPE;
    if (ffn_workspace_bytes(M, I) > kFfnStaticScratchBytes) return NVFP4_ERR_UNSUPPORTED;
    int dev = 0;
    const cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return cuda_fail(e);
    void* ws = ffn_static_scratch(dev, static_cast<cudaStream_t>(stream));
    if (!ws) return cuda_fail(cudaGetLastError());
    return nvfp4_ffn_swiglu(w_gate, s_gate, g_gate, w_up, s_up, g_up, w_down, s_down, g_down, x, clamp_limit, ws, y,
                            y_type, M, H, I, stream);
}

nvfp4_status nvfp4_moe_gemv(const uint8_t* w_packed, const uint8_t* w_scales,
                            const float* global_scales, int E,
                            const int32_t* expert_ids, int T, int top_k,
                            const uint16_t* x, int x_per_slot,
                            void* y, nvfp4_out_t y_type, int N, int K,
                            int32_t* status_dev, void* stream) {
    if (!w_packed || !w_scales || !global_scales || !expert_ids || !x || !y) return NVFP4_ERR_NULL;
    if (E < 1 || T < 0 || top_k < 0 || N < 0 || K < 0 || K % 16 != 0) return NVFP4_ERR_SHAPE;
    if (static_cast<int64_t>(T) * top_k > (1 << 24)) return NVFP4_ERR_UNSUPPORTED;
    const nvfp4_status so = check_out(y_type);
    if (so != NVFP4_OK) return so;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int slots = T * top_k;
    if (slots == 0 || N == 0) return NVFP4_OK;
    if (K == 0) return zero_output(y, static_cast<int64_t>(slots) * N, y_type, st);
    int dev = 0;
    const DeviceInfo* d = device_info(&dev);
    if (!d) return cuda_fail(cudaGetLastError());
    if (slots <= kMaxMoeSlots && static_cast<int64_t>(E) * N <= (1 << 30)) {
        // warp-tile kernel: every routed expert's slab is read once for up to 8 of its slots
        // (more than 32 slots: the stream-K form only)
        TilePlan tpl{};
        const uint8_t* wv[1] = {w_packed};
        const uint8_t* sv[1] = {w_scales};
        const int xrows = x_per_slot ? slots : T;
        const bool x_ok = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
        const PlanKey key = make_key(dev, 5 + (x_ok ? 0 : 8), 8, N, K, 1, wv, sv, E, T, top_k, x_per_slot ? 1 : 0);
        const bool tile = cached_tile_plan(key, &tpl, [&](TilePlan& tp) {
            if (!plan_tile(tp, 8, N, K, expected_groups(E, T, top_k), *d, wv, sv, x, true, xrows, slots)) return false;
            if (!encode_tile_maps(&tp.p.wmap[0], &tp.p.smap[0], w_packed, w_scales, static_cast<int64_t>(E) * N, K,
                                  tp.nc))
                return false;
            tp.p.wmap[1] = tp.p.wmap[0];
            tp.p.smap[1] = tp.p.smap[0];
            return true;
        });
        if (tile) {
            TileParams& p = tpl.p;
            p.x = x;
            p.y = y;
            p.ldy = N;
            p.out_bf16 = y_type == NVFP4_OUT_BF16;
            p.force_f32 = g_variant == 2;
            p.wait_ns = g_wait_ns;
            p.ids = expert_ids;
            p.g_dev = global_scales;
            p.status_user = status_dev;
            p.E = E;
            p.top_k = top_k;
            p.slots = slots;
            p.x_per_slot = x_per_slot ? 1 : 0;
            const cudaError_t e = launch_tile(tpl, st, true);
            if (e != cudaSuccess) return cuda_fail(e);
            const cudaError_t e2 = cudaGetLastError();
            return e2 == cudaSuccess ? NVFP4_OK : cuda_fail(e2);
        }
    }
    Plan pl{};
    if (plan_moe(pl, E, T, top_k, N, K, *d, w_packed, w_scales, x)) {
        Params& p = pl.p;
        p.w[0] = p.w[1] = w_packed;
        p.s[0] = p.s[1] = w_scales;
        p.g_dev = global_scales;
        p.ids = expert_ids;
        p.status_user = status_dev;
        p.x = x;
        p.x_per_slot = x_per_slot ? 1 : 0;
        p.y = y;
        p.ldy = N;
        p.out_bf16 = y_type == NVFP4_OUT_BF16;
        p.M = 1;
        p.wait_ns = g_wait_ns;
        p.force_f32 = g_variant == 2;
        const cudaError_t e = dispatch_stream(pl, st);
        if (e != cudaSuccess) return cuda_fail(e);
        const cudaError_t e2 = cudaGetLastError();
        return e2 == cudaSuccess ? NVFP4_OK : cuda_fail(e2);
    }
    SimpleParams sp{};
    sp.w[0] = sp.w[1] = w_packed;
    sp.s[0] = sp.s[1] = w_scales;
    sp.g_dev = global_scales;
    sp.ids = expert_ids;
    sp.status_user = status_dev;
    sp.x = x; sp.y = y; sp.ldy = N; sp.out_bf16 = y_type == NVFP4_OUT_BF16;
    sp.M = 1; sp.N = N; sp.K = K; sp.groups = 1;
    sp.moe = 1; sp.E = E; sp.top_k = top_k; sp.x_per_slot = x_per_slot ? 1 : 0; sp.slots = slots;
    const cudaError_t e = launch_simple(sp, static_cast<int64_t>(slots) * N, st);
    return e == cudaSuccess ? NVFP4_OK : cuda_fail(e);
}

const char* nvfp4_status_string(int status) {
    switch (status) {
        case NVFP4_OK: return "ok";
        case NVFP4_ERR_NULL: return "null pointer";
        case NVFP4_ERR_SHAPE: return "invalid shape (need 0<=M<=8, N>=0, K>=0, K%16==0)";
        case NVFP4_ERR_ALIGN: return "misaligned pointer";
        case NVFP4_ERR_DTYPE: return "invalid output type";
        case NVFP4_ERR_UNSUPPORTED: return "unsupported size";
        case NVFP4_ERR_CUDA: return "CUDA runtime error";
        case NVFP4_ERR_TIMEOUT: return "device pipeline wait timed out";
        default: return "unknown status";
    }
}

int nvfp4_last_cuda_error(void) { return g_last_cuda_error; }

nvfp4_status nvfp4_device_status(int32_t* flags_out, void* stream) {
    if (!flags_out) return NVFP4_ERR_NULL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    int v = 0;
    cudaError_t e = cudaStreamSynchronize(st);
    if (e != cudaSuccess) return cuda_fail(e);
    e = cudaMemcpyFromSymbol(&v, g_device_status, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
    const int zero = 0;
    e = cudaMemcpyToSymbol(g_device_status, &zero, sizeof(int));
    if (e != cudaSuccess) return cuda_fail(e);
    *flags_out = v;
    return (v & NVFP4_DEV_TIMEOUT) ? NVFP4_ERR_TIMEOUT : NVFP4_OK;
}

void nvfp4_set_wait_budget_ns(uint64_t ns) { g_wait_ns = ns == UINT64_MAX ? kDefaultWaitNs : ns; }

void nvfp4_set_variant(int variant) { g_variant = variant; }

void nvfp4_set_pdl(int enable) { g_pdl = enable != 0; }

int nvfp4_phase_trace(uint64_t* host_out, int max_words, void* stream) {
#if NVFP4_PHASE_TRACE
    if (!host_out || max_words < 0) return -1;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
    const int total = kTraceLaunches * kTraceCtas * kTraceWords;
    const int n = std::min(total, max_words);
    if (n > 0 && cudaMemcpyFromSymbol(host_out, g_trace, static_cast<size_t>(n) * 8) != cudaSuccess) return -1;
    void* dev = nullptr;
    if (cudaGetSymbolAddress(&dev, g_trace) != cudaSuccess) return -1;
    if (cudaMemset(dev, 0, static_cast<size_t>(total) * 8) != cudaSuccess) return -1;
    if (cudaDeviceSynchronize() != cudaSuccess) return -1;
    {
        std::lock_guard<std::mutex> lk(g_mu);
        g_trace_next = 0;
    }
    return n;
#else
    (void)host_out; (void)max_words; (void)stream;
    return 0;
#endif
}

long long nvfp4_fp32_fallbacks(void* stream) {
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    unsigned long long v = 0;
    if (cudaStreamSynchronize(st) != cudaSuccess) return -1;
    if (cudaMemcpyFromSymbol(&v, g_fp32_fallbacks, sizeof v) != cudaSuccess) return -1;
    const unsigned long long zero = 0;
    if (cudaMemcpyToSymbol(g_fp32_fallbacks, &zero, sizeof zero) != cudaSuccess) return -1;
    return static_cast<long long>(v);
}

}  // extern "C"

namespace nvfp4 {

// The launch a call would make on device d; host_only: the tile kernel's tensor-map encoder
// (a driver entry point) is assumed present, so no GPU or driver is needed.
int describe_plan_on(const DeviceInfo* d, bool host_only, int kind, int M, int N, int K, int T, int top_k,
                     char* buf, int buflen) {
    Plan pl{};
    bool ok = false;
    // Pointers are only inspected for alignment here; 256-byte aligned stand-ins.
    const uint8_t* fake = reinterpret_cast<const uint8_t*>(static_cast<uintptr_t>(256));
    const uint8_t* w[2] = {fake, fake};
    if (kind == 5) {  // dense with dictionary scales: the tile kernel's SD form, else the byte-load kernel
        TilePlan tpl{};
        if (K % 256 == 0 && plan_tile(tpl, M, N, K, 1, *d, w, w, fake, false, 0, 0, false, !host_only, true))
            return snprintf(buf, buflen,
                            "tile_sdict grid=%d block=%d smem=%u split=%d rows_per_item=%d k_warps=%d mt=%d stages=%d nc=%d",
                            tpl.grid_x * tpl.grid_y, tk::kThreads, tpl.smem, 1 << tpl.p.s_log2, tpl.p.tpi * 16,
                            1 << tpl.p.ksplit_log2, M, tpl.p.stages, tpl.nc);
        return snprintf(buf, buflen, "simple grid=%lld block=%d smem=0 split=1 rows_per_item=0 k_warps=0",
                        static_cast<long long>((static_cast<int64_t>(N) + 7) / 8), kSimpleThreads);
    }
    if (kind == 6 || kind == 7) {  // MoE with dictionary scales (M = E; 7: one x row per slot)
        TilePlan tpl{};
        const int slots = T * top_k, E = M;
        const int xrows = kind == 7 ? slots : T;
        if (K % 256 == 0 && slots <= kMaxMoeSlots && E >= 1 && static_cast<int64_t>(E) * N <= (1 << 30) &&
            plan_tile(tpl, 8, N, K, expected_groups(E, T, top_k), *d, w, w, fake, true, xrows, slots, false,
                      !host_only, true) &&
            tpl.sk && tpl.p.items_r)
            return snprintf(buf, buflen,
                            "tile_sk_moe_sdict grid=%d block=%d smem=%u split=1 rows_per_item=%d k_warps=1 mt=8 "
                            "stages=%d nc=%d group_aligned=1",
                            tpl.grid_x, tk::kThreads, tpl.smem, tpl.p.tpi * 16, tpl.p.stages, tpl.nc);
        return snprintf(buf, buflen, "simple grid=%lld block=%d smem=0 split=1 rows_per_item=0 k_warps=0",
                        static_cast<long long>((static_cast<int64_t>(slots) * N + 7) / 8), kSimpleThreads);
    }
    if (kind == 8) {  // the FFN block (N = H, K = I): one fused launch, else gate/up + activation, then down
        FfnPlan fp{};
        if (N % 16 == 0 && K % 16 == 0 && plan_ffn(fp, M, N, K, *d) &&
            (host_only || (fp.nc == 2 ? ffn_two_per_sm<2>(fp.smem) : ffn_two_per_sm<1>(fp.smem))))
            return snprintf(buf, buflen,
                            "ffn_fused grid=%d block=%d smem=%u split=1 rows_per_item=%d k_warps=%d mt=%d stages=%d "
                            "nc=%d down_rows_per_item=%d down_k_warps=%d",
                            fp.grid, tk::kThreads, fp.smem, fp.p.a.tpi * 16, 1 << fp.p.a.ksplit_log2, M,
                            fp.p.a.stages, fp.nc, fp.p.b.tpi * 16, 1 << fp.p.b.ksplit_log2);
        char a[200], b[200];
        describe_plan_on(d, host_only, 4, M, K, N, 0, 0, a, sizeof a);
        describe_plan_on(d, host_only, 0, M, N, K, 0, 0, b, sizeof b);
        return snprintf(buf, buflen, "ffn_two_launch gate_up=[%s] down=[%s]", a, b);
    }
    if (kind == 4) {  // gate/up with the fused activation: the tile kernel, else the byte-load kernel
        TilePlan tpl{};
        if (plan_tile(tpl, M, N, K, 2, *d, w, w, fake, false, 0, 0, true, !host_only))
            return snprintf(buf, buflen,
                            "tile_swiglu grid=%d block=%d smem=%u split=%d rows_per_item=%d k_warps=%d mt=%d stages=%d nc=%d",
                            tpl.grid_x * tpl.grid_y, tk::kThreads, tpl.smem, 1 << tpl.p.s_log2, tpl.p.tpi * 16,
                            1 << tpl.p.ksplit_log2, M, tpl.p.stages, tpl.nc);
        return snprintf(buf, buflen, "simple grid=%lld block=%d smem=0 split=1 rows_per_item=0 k_warps=0",
                        static_cast<long long>((static_cast<int64_t>(N) + 7) / 8), kSimpleThreads);
    }
    if (kind == 0 || kind == 1) {
        TilePlan tpl{};
        if (plan_tile(tpl, M, N, K, kind == 0 ? 1 : 2, *d, w, w, fake, false, 0, 0, false, !host_only)) {
            return snprintf(buf, buflen,
                            "tile grid=%d block=%d smem=%u split=%d rows_per_item=%d k_warps=%d mt=%d stages=%d nc=%d",
                            tpl.grid_x * tpl.grid_y, tk::kThreads, tpl.smem, 1 << tpl.p.s_log2, tpl.p.tpi * 16,
                            1 << tpl.p.ksplit_log2, M, tpl.p.stages,
                            tpl.nc);
        }
        ok = plan_dense(pl, M, N, K, kind == 0 ? 1 : 2, *d, w, w, fake);
    }
    if (kind == 2 || kind == 3) {
        // MoE: M is the number of experts E; kind 3 has one x row per slot
        TilePlan tpl{};
        const int slots = T * top_k, E = M;
        const int xrows = kind == 3 ? slots : T;
        if (slots <= kMaxMoeSlots && E >= 1 && static_cast<int64_t>(E) * N <= (1 << 30) &&
            plan_tile(tpl, 8, N, K, expected_groups(E, T, top_k), *d, w, w, fake, true, xrows, slots, false,
                      !host_only)) {
            return snprintf(buf, buflen,
                            "%s grid=%d block=%d smem=%u split=1 rows_per_item=%d k_warps=%d mt=8 stages=%d nc=%d "
                            "group_aligned=%d",
                            tpl.sk ? "tile_sk_moe" : "tile_moe", tpl.grid_x, tk::kThreads, tpl.smem, tpl.p.tpi * 16,
                            1 << tpl.p.ksplit_log2, tpl.p.stages, tpl.nc, tpl.sk ? tpl.p.items_r : 0);
        }
        ok = plan_moe(pl, E, T, top_k, N, K, *d, fake, fake, fake);
    }
    int n;
    if (!ok) {
        n = snprintf(buf, buflen, "simple grid=%lld block=%d smem=0 split=1 rows_per_item=0 k_warps=0",
                     static_cast<long long>(((kind >= 2 ? static_cast<int64_t>(T) * top_k : (kind == 1 ? 2 : 1)) * N + 7) / 8),
                     kSimpleThreads);
    } else {
        n = snprintf(buf, buflen, "%s grid=%d block=%d smem=%u split=%d rows_per_item=%d k_warps=%d mt=%d stages=%d",
                     pl.kind == 1 ? "stream_moe" : "stream", pl.grid, kThreads, pl.smem, pl.p.S, pl.p.rpi,
                     pl.p.ck, pl.mt, pl.p.stages);
    }
    return n;
}

}  // namespace nvfp4

extern "C" {

int nvfp4_describe_plan(int kind, int M, int N, int K, int T, int top_k, char* buf, int buflen) {
    if (!buf || buflen < 1) return -1;
    const DeviceInfo* d = device_info(nullptr);
    if (!d) return -1;
    return describe_plan_on(d, false, kind, M, N, K, T, top_k, buf, buflen);
}

int nvfp4_describe_plan_host(int sm_count, int smem_optin, int smem_per_sm, int kind, int M, int N, int K, int T,
                             int top_k, char* buf, int buflen) {
    if (!buf || buflen < 1 || sm_count < 1 || smem_optin < 1 || smem_per_sm < smem_optin) return -1;
    if (kind < 0 || kind > 8) return -1;
    DeviceInfo d;
    d.sm_count = sm_count;
    d.smem_optin = smem_optin;
    d.smem_per_sm = smem_per_sm;
    d.init = true;
    return describe_plan_on(&d, true, kind, M, N, K, T, top_k, buf, buflen);
}

int nvfp4_version(void) { return 100; }

}  // extern "C"
