// internal.cuh -- shared definitions of the sm_103a kernels and the host runtime.
// Not part of the public ABI (include/rwkv7.h is).
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace rk {

// ----------------------------------------------------------------------------
// Device error word bits (latched by kernels, read by rwkv7_synchronize).
// ----------------------------------------------------------------------------
enum : uint32_t {
    ERR_SLOT = 1u,     // slot index out of range
    ERR_TOKEN = 2u,    // token id out of range
    ERR_DUP = 4u,      // a slot appears twice in one step
    ERR_TIMEOUT = 8u,  // a bounded wait gave up
    ERR_CONFIG = 16u,  // the sampler found no token to draw (no finite weight)
};

constexpr int HS = 64;             // head size
constexpr int MAX_B = 256;         // slots per fused step
constexpr int GEMM_TILE_M = 128;   // weight rows per tile (MMA M)
constexpr int GEMM_TILE_K = 64;    // reduction elements per stage (128 bytes of fp16)
constexpr int GEMM_MAX_SEG = 12;
constexpr int GEMM_MAX_MAPS = 24;
constexpr int MAX_SPLIT = 16;         // k-splits of one projection
constexpr uint64_t WAIT_LIMIT_NS = 2000000000ull;  // bounded waits give up after ~2 s

// Epilogue kinds of the projection GEMM.  acc is the fp32 dot product of one
// weight row n with one activation row b.
enum Epi : int {
    EPI_F32 = 0,         // out f32 = acc
    EPI_F16 = 1,         // out f16 = acc
    EPI_F16_TANH = 2,    // out f16 = tanh(acc)
    EPI_F16_SIGMOID = 3, // out f16 = sigmoid(acc)
    EPI_DECAY = 4,       // out f32 = exp(-exp(-1/2) * sigmoid(bias[n] + acc))
    EPI_SIGMOID_BIAS = 5,// out f32 = sigmoid(bias[n] + acc)
    EPI_RESID = 6,       // out f32 += acc (residual stream)
    EPI_RELU2 = 7,       // out f16 = relu(acc)^2, plus a nonzero flag per 64 rows
};

// One weight matrix of a projection launch.  Weights are stored tile-major:
// tile (row block tr, k-block kb) of 128 rows x 64 k fp16 is 16 KB contiguous,
// tiles ordered (layer, tr, kb); ragged rows / k are zero-padded.  A segment's
// row tiles are split into S contiguous k-ranges ("items"): S == 1 applies the
// epilogue, S > 1 stores raw fp32 partial sums, slab j at out + j*split_stride,
// which the consuming kernel adds in slab order.
struct GemmSeg {
    int wmap, xmap;       // tensor-map indices (tensor-core path)
    int x3;               // 1: xmap is the 3D (col, row, k-block) view, one copy per stage
    int tile_base;        // map tile index of (this layer, row tile 0, k-block 0)
    int rows, K, kb;      // output rows, reduction length, k-blocks of 64
    int tiles, S;         // row tiles, k-splits
    int item0;            // first global item of this segment
    int epi;
    void *out;
    int ldo;              // out element index = b * ldo + n (+ j * split_stride)
    long long split_stride;
    const __half *bias;   // [rows] (EPI_DECAY / EPI_SIGMOID_BIAS)
    const __half *wscale; // int8 weights: fp16 scale per output row (applied to the sum), else null
    const __half *w;      // tiled weights of this layer (SIMT path)
    const __half *x;      // activations [B][ldx] (SIMT path)
    int ldx;
    // Split segment finished in the launch (two-phase launches): each row
    // tile's last item to store its partial slab adds the S slabs in slab
    // order, applies fix_epi (an fp16 kind) and stores the result at fix_out
    // (element b * ldo + n).  fix_ctr: one counter per row tile, zero at
    // launch.  Null fix_out: the consumer adds the slabs.
    void *fix_out;
    uint32_t *fix_ctr;
    int fix_epi;
};

struct GemmParams {
    CUtensorMap maps[GEMM_MAX_MAPS]; // weight and activation maps used by the segments
    GemmSeg seg[GEMM_MAX_SEG];
    int nseg, nmaps, nitems;
    int B, npad;                     // slots in the step, MMA N (B rounded up to 16)
    int stages;                      // smem pipeline depth (int8 weights: stages of the int8 + activation ring)
    int stages_b;                    // int8 weights: stages of widened weights in tensor memory
    int stages_x;                    // int8 weights: stages of the activation ring
    int kbs;                         // int8 weights: k-blocks per stage (1 or 2); fp16 weights: always 2
    int accbufs;                     // TMEM accumulator buffers (1 or 2)
    int prefetch;                    // weight stages that may be fetched before the dependency wait (0: none)
    uint32_t *nz_out;                // EPI_RELU2: flag per 64 output rows
    unsigned long long *nz_count;    // EPI_RELU2: running count of nonzero 64-row blocks (or null)
    const uint32_t *nz_skip;         // nonzero flags per k-block of the activations (or null)
    uint32_t *err;
    unsigned long long *tl;          // timeline words of this launch (measurement only; else null)
    // Two-phase launch: items [0, n0) (the first segments) are phase 0, spread
    // over CTAs [0, g0); the rest are phase 1, spread over CTAs [0, p1a) and
    // [p1b, grid), and their activations -- produced by the phase-0 items
    // [0, ndep) -- are read only once *dep (zero at launch) reaches dep_target:
    // each stored unsplit item of [0, ndep) adds one, each row tile of a split
    // segment finished in the launch (GemmSeg::fix_out) one.  Phase-0 items
    // past ndep feed no phase-1 item and run beside the chain.  Every CTA must
    // be resident at once: the grid is at most one CTA per SM.  n0 = 0: one
    // phase (p1a = p1b = 0).
    int n0, g0, ndep, dep_target, p1a, p1b;
    uint32_t *dep;
    int skip_seg;                    // segment whose activations nz_skip describes
};

// Raise a kernel's dynamic shared-memory limit on the current device, once per
// (kernel, device, size); thread-safe (a process may drive several devices).
cudaError_t ensure_smem_attr(const void *kernel, int bytes);

// Launch helpers (implemented in the .cu files).
struct LaunchCfg {
    cudaStream_t stream;
    bool pdl;   // programmatic dependent launch
};

void launch_gemm_tc(const GemmParams &p, int grid, size_t smem, const LaunchCfg &lc, cudaError_t *e);
void launch_gemm_simt(const GemmParams &p, const LaunchCfg &lc, cudaError_t *e);
size_t gemm_tc_smem_bytes(int npad, int stages);
// int8-weight GEMM: weights arrive as int8 tiles and are converted to fp16 in
// shared memory by the epilogue warps before the tensor cores read them.
void launch_gemm_tc8(const GemmParams &p, int grid, size_t smem, const LaunchCfg &lc, cudaError_t *e);
size_t gemm_tc8_smem_bytes(int npad, int kbs, int stages_w, int stages_x);
size_t gemm_tc_stage_bytes(int npad);
int gemm_tc_max_smem();

struct ElemParams {
    int B, d, H, F, V, n_slots, layer, L;
    const int32_t *slots, *tokens;
    float *x;                 // residual [B][d]
    const __half *emb;        // [V][d]
    const __half *ln_w, *ln_b;
    const __half *mu[6];      // token-shift mixes
    __half *xo[6];            // mixed outputs [B][d]
    float *shift;             // shift state base of this layer [n_slots][d]
    const float *part;        // residual partial slabs to add to x first (or null)
    int nsplit;
    long long split_stride;
    uint32_t *err;
    int single_slot;          // prefill: every row is a token of this slot (-1: rows are slots)
    float *xout;              // prefill: residual after the slab adds (x is read only)
    unsigned long long *tl;   // timeline words of this launch (measurement only; else null)
};

void launch_embed(const ElemParams &p, const LaunchCfg &lc, cudaError_t *e);
// Prefill of one slot: rows are the consecutive tokens of a chunk.  The token
// shift takes the previous row's LayerNorm output (the slot's shift state for
// row 0) and leaves the last row's in the shift state.
void launch_ln_mix_prefill(const ElemParams &p, int nmix, const LaunchCfg &lc, cudaError_t *e);

// Prefill WKV of one slot over n tokens, in three kernels:
//  vectors per (token, head): kh, kh*a, kp, vp, r and the bonus scalar;
//  the sequential state update (4 CTAs per head, 16 state rows each): y;
//  GroupNorm + bonus + output gate: z.
struct WkvSeqParams {
    int n, d, H, slot, n_slots, layer;
    const float *r, *k, *v;          // projection split slabs [nsplit][bcap][d]
    int nsplit;
    long long split_stride;
    const float *dec, *a, *vg, *g;   // [n][d]
    float *v_first;                  // [n][d]
    const __half *k_k, *k_a, *r_k, *lnx_w, *lnx_b;
    float *vec;                      // per-head vectors [H][vec_rows][6][64]: kh, kh*a, dec, kp, r, vp
    int vec_rows;
    float *bonus, *y;                // [n][H], [n][d]
    float *wkv;                      // this layer's states [n_slots][H][64][64]
    __half *z;                       // [n][d]
    uint32_t *err;
};
void launch_wkv_prefill(const WkvSeqParams &p, const LaunchCfg &lc, cudaError_t *e);
void launch_ln_mix(const ElemParams &p, int nmix, const LaunchCfg &lc, cudaError_t *e);
void launch_ln_out(const ElemParams &p, const LaunchCfg &lc, cudaError_t *e);


struct WkvParams {
    int B, d, H, n_slots, layer;
    const int32_t *slots;
    const float *r, *k, *v;          // projection partial slabs [nsplit][bcap][d]
    int nsplit;
    long long split_stride;
    const float *dec, *a, *vg, *g;   // gates from the LoRA-up projection, [B][d]
    float *v_first;                  // [B][d]
    const __half *k_k, *k_a, *r_k, *lnx_w, *lnx_b;
    float *wkv;                      // this layer's states [n_slots][H][64][64]
    __half *z;                       // [B][d]
    uint32_t *err;
    unsigned long long *tl;          // timeline words of this launch (measurement only; else null)
};
void launch_wkv(const WkvParams &p, const LaunchCfg &lc, cudaError_t *e);

// LoRA-down outputs: add the S partial slabs, apply the activation (0 none,
// 1 tanh, 2 sigmoid), round to fp16.  r[i] == 0 skips LoRA i.
struct LoraFinParams {
    int B, S, bcap;
    int r[4];
    int act[4];
    const float *part[4];  // [S][bcap][r]
    __half *out[4];        // [B][r]
    unsigned long long *tl;  // timeline words of this launch (measurement only; else null)
};
void launch_lora_fin(const LoraFinParams &p, const LaunchCfg &lc, cudaError_t *e);

struct SampleParamsDev {  // device copy of one slot's sampling parameters
    float temperature, top_p;
    int32_t top_k;
    float presence, frequency, penalty_decay;
    unsigned long long seed;
    int32_t greedy, pad;
};

struct SamplerParams {
    int B, V, n_slots;
    const int32_t *slots;
    const float *logits;   // [B][V]
    float *occ;            // [n_slots][V]
    const SampleParamsDev *params;  // [n_slots]
    unsigned long long *ndraw;      // [n_slots]
    float *lpen;           // scratch [B][V]
    int32_t *next;         // [B]
    uint32_t *err;
    unsigned long long *tl;  // timeline words of this launch (measurement only; else null)
};
void launch_sampler(const SamplerParams &p, const LaunchCfg &lc, cudaError_t *e);

struct SlotOpParams {
    int op;  // 0 reset, 1 copy src->dst, 2 swap
    int a, b;
    int L, n_slots;
    size_t wkv_per_slot;   // floats per slot per layer
    size_t d;              // shift floats per slot per layer
    int V;
    float *wkv, *shift_att, *shift_ffn, *occ;
    unsigned long long *ndraw;
    SampleParamsDev *params;
};
void launch_slot_op(const SlotOpParams &p, cudaStream_t s, cudaError_t *e);

}  // namespace rk

// ----------------------------------------------------------------------------
// Device-side PTX helpers.
// ----------------------------------------------------------------------------
#ifdef __CUDACC__
namespace rk {

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ uint64_t gtimer() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// In-graph timeline of a step (a measurement aid; the pointer is null in normal
// steps).  Each launch owns four %globaltimer words: the earliest CTA start,
// the earliest and latest return from the dependency wait, the latest CTA end.
// Start words are preset to all ones, the others to zero.
__device__ __forceinline__ void tl_start(unsigned long long *tl) {
    if (tl) atomicMin(tl, (unsigned long long)gtimer());
}
__device__ __forceinline__ void tl_release(unsigned long long *tl) {
    if (tl) {
        const unsigned long long t = gtimer();
        atomicMin(tl + 1, t);
        atomicMax(tl + 2, t);
    }
}
__device__ __forceinline__ void tl_end(unsigned long long *tl) {
    if (tl) atomicMax(tl + 3, (unsigned long long)gtimer());
}

// Programmatic dependent launch: wait for the preceding grid's completion (and
// memory), and allow the next grid to be scheduled.  No-ops without PDL.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}
// Bounded wait for the phase with `parity`.  Gives up (returns false) after
// WAIT_LIMIT_NS or as soon as *abort is non-zero.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, volatile uint32_t *abort) {
    if (mbar_try_wait(bar, parity)) return true;
    uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (*abort) return false;
            if (gtimer() - t0 > WAIT_LIMIT_NS) return false;
        }
    }
}

// Bounded wait that ignores the abort word: used to drain copies still in
// flight before a CTA exits, when the abort word may already be set.
__device__ __forceinline__ bool mbar_wait_any(uint64_t *bar, uint32_t parity) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = gtimer();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0 && gtimer() - t0 > WAIT_LIMIT_NS) return false;
    }
}
__device__ __forceinline__ void fence_barrier_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// Contiguous bulk copies between global and shared memory (16-byte aligned,
// size a multiple of 16).
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}
__device__ __forceinline__ void bulk_s2g(void *dst, const void *src, uint32_t bytes) {
    asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst), "r"(smem_u32(src)),
                 "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void prefetch_tmap(const CUtensorMap *m) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(m) : "memory");
}

// TMA tiled loads into shared memory, completing transaction bytes on `bar`.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0, int c1,
                                            uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3}], [%4], %5;" ::"r"(smem_u32(dst)),
        "l"(m), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}
__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *m, uint64_t *bar, int c0, int c1,
                                            int c2, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
        " [%0], [%1, {%2, %3, %4}], [%5], %6;" ::"r"(smem_u32(dst)),
        "l"(m), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// ---- tcgen05 (5th-generation tensor cores, accumulators in tensor memory) ----
__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]^T, fp16 inputs, fp32 accumulate.
__device__ __forceinline__ void mma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive on `bar` once every previously issued tcgen05.mma of this thread completes.
// D[tmem] (+)= A[tmem] * B[smem]^T, fp16 inputs, fp32 accumulate: A (M = 128
// rows) read from tensor memory, row m in lane m, fp16 elements (2j, 2j + 1)
// of its K slice packed in column j (low half first).
__device__ __forceinline__ void mma_f16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                           uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// 32 lanes x 32 columns of 32-bit values from registers into tensor memory
// (lane i of the warp -> TMEM lane base + i, register j -> column base + j).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]),
        "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]),
        "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]),
        "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void mma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                     smem_u32(bar))
                 : "memory");
}
// 32 lanes x 16 / 32 columns of 32-bit accumulator words: lane i of the warp
// gets TMEM lane (base lane + i), columns [col, col + 16 / 32).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
    uint32_t r[32];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, "
        "%14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
          "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
          "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor of a K-major operand tile stored as rows of
// 128 bytes (64 fp16) with the 128-byte swizzle, 8-row groups 1024 bytes apart.
__device__ __forceinline__ uint64_t sdesc_k128(uint32_t saddr) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);   // start address
    d |= (uint64_t)1 << 16;                       // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024 >> 4) << 32;             // stride byte offset: next 8-row group
    d |= (uint64_t)1 << 46;                       // descriptor version (sm_100 family)
    d |= (uint64_t)2 << 61;                       // 128-byte swizzle
    return d;
}

// Instruction descriptor: kind::f16 with fp16 A/B, fp32 D, both K-major.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N) {
    return (1u << 4) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// Activations of the gate epilogues with the hardware exp2 / reciprocal paths
// (__expf, __fdividef).  Their error (a few ulp of fp32) is far below what the
// fp16 rounding of the LoRA hidden vectors and the model tolerance allow.
__device__ __forceinline__ float fast_sigmoid(float x) { return __fdividef(1.0f, 1.0f + __expf(-x)); }
__device__ __forceinline__ float fast_tanh(float x) {
    // tanh x = 1 - 2 / (1 + e^{2x}); near 0 the series x - x^3/3 avoids cancellation
    if (fabsf(x) < 0.03125f) return x - x * x * x * (1.0f / 3.0f);
    return 1.0f - __fdividef(2.0f, 1.0f + __expf(2.0f * x));
}
// RWKV-7 decay from the LoRA output: exp(-e^{-1/2} * sigmoid(w))
__device__ __forceinline__ float rwkv_decay(float w) { return __expf(-0.606530659712633f * fast_sigmoid(w)); }

__device__ __forceinline__ void named_bar(int id, int nthreads) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

}  // namespace rk
#endif
