// rwkv7_api.cu -- host runtime behind include/rwkv7.h: device weights, the slot
// pool, activation buffers, TMA descriptors, the per-step launch sequence and
// its CUDA-graph cache.
//
// One decode step of B slots (RWKV-Runner Albatross article, "连续批处理Worker
// 主循环": forward_seq_batch then sample_next_tokens_batch) launches
//   embed+LN0 | per layer: LN1+mix6, G1 (r,k,v + LoRA down), G2 (LoRA up +
//   gates), WKV7+GroupNorm+gate, G3 (output + residual), LN2+mix, G4 (key,
//   ReLU^2), G5 (value + residual, skipping all-zero hidden blocks) |
//   LN_out, head, sampler
// with programmatic dependent launch between kernels so each kernel's weight
// prefetch overlaps its predecessor's tail, replayed from a CUDA graph per
// (B, head, sampling) combination.
#include <cudaTypedefs.h>

#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <map>
#include <mutex>
#include <string>
#include <tuple>
#include <vector>

#include "../../include/rwkv7.h"
#include "internal.cuh"

using namespace rk;

cudaError_t rk::ensure_smem_attr(const void *kernel, int bytes) {
    // The kernel's dynamic shared-memory limit on the current device is raised
    // to the largest size asked for so far and never lowered (a launch of a
    // smaller size fits under it; lowering it would break a later, larger
    // launch that the table already counts as set).  A fixed table (no heap
    // allocation, so the allocation-free sampler path can use it); when it is
    // full the attribute is simply set again on every call.
    struct Entry {
        const void *kernel;
        int dev, bytes;
    };
    static std::mutex mu;
    static Entry done[256];
    static int ndone = 0;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lk(mu);
    int at = -1;
    for (int i = 0; i < ndone; ++i)
        if (done[i].kernel == kernel && done[i].dev == dev) {
            if (done[i].bytes >= bytes) return cudaSuccess;
            at = i;
        }
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e != cudaSuccess) return e;
    if (at >= 0)
        done[at].bytes = bytes;
    else if (ndone < 256)
        done[ndone++] = Entry{kernel, dev, bytes};
    return cudaSuccess;
}

namespace {

// ---------------------------------------------------------------- weights
enum WK {
    W_EMB, W_HEAD, W_LN0W, W_LN0B, W_LNOW, W_LNOB,
    L_LN1W, L_LN1B, L_LN2W, L_LN2B,
    L_XR, L_XW, L_XK, L_XV, L_XA, L_XG,
    L_W0, L_W1, L_W2, L_A0, L_A1, L_A2, L_V0, L_V1, L_V2, L_G1, L_G2,
    L_KK, L_KA, L_RK, L_WR, L_WK, L_WV, L_WO, L_LNXW, L_LNXB,
    L_FXK, L_FK, L_FV, W_COUNT
};
constexpr int FIRST_LAYER_KIND = L_LN1W;

const char *kind_name[W_COUNT] = {
    "emb", "head", "ln0.w", "ln0.b", "ln_out.w", "ln_out.b",
    "ln1.w", "ln1.b", "ln2.w", "ln2.b",
    "att.x_r", "att.x_w", "att.x_k", "att.x_v", "att.x_a", "att.x_g",
    "att.w0", "att.w1", "att.w2", "att.a0", "att.a1", "att.a2", "att.v0", "att.v1", "att.v2", "att.g1", "att.g2",
    "att.k_k", "att.k_a", "att.r_k", "att.receptance", "att.key", "att.value", "att.output", "att.ln_x.w",
    "att.ln_x.b", "ffn.x_k", "ffn.key", "ffn.value"};

// kernel classes reported by rwkv7_profile_step
enum PClass { P_EMBED, P_LN_MIX, P_GEMM_PROJ, P_GEMM_LORA, P_WKV, P_GEMM_OUT, P_GEMM_KEY, P_GEMM_VALUE, P_LN_OUT,
              P_GEMM_HEAD, P_SAMPLER, P_LORA_FIN, P_GEMM_FFN, P_COUNT };

struct Prof {
    std::vector<cudaEvent_t> ev;  // pairs (begin, end)
    std::vector<int> cls;
    size_t n = 0;
};

// activation buffers addressed by tensor maps
enum ABuf { A_XR, A_XW, A_XK, A_XV, A_XA, A_XG, A_HW, A_HA, A_HV, A_HG, A_Z, A_XKF, A_H, A_XO, A_COUNT };

// Device allocator for contexts created from now on (rwkv7_set_device_allocator);
// both null: cudaMalloc / cudaFree.
struct DevAllocator {
    rwkv7_alloc_fn alloc = nullptr;
    rwkv7_free_fn release = nullptr;
    void *user = nullptr;
};
std::mutex g_alloc_mu;
DevAllocator g_alloc;

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    if (!fn) {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
    }
    return fn;
}

}  // namespace

struct rwkv7_ctx {
    rwkv7_config cfg{};
    int L = 0, d = 0, H = 0, F = 0, V = 0, rw = 0, ra = 0, rv = 0, rg = 0, n_slots = 0;
    int bcap = 0;  // activation rows (max slots per fused step, rounded up to 16)
    int nsm = 0;
    cudaStream_t stream = nullptr;      // caller's stream: every call is ordered on it
    cudaStream_t cap_stream = nullptr;  // private stream used only to capture step graphs
    int mode = 0;
    std::string err;

    // weights: vectors and the embedding row-major; projection matrices tile-major
    // (tiled[k]: [layer][row tile][k-block][128][64] fp16, zero-padded)
    int wrows[W_COUNT]{}, wcols[W_COUNT]{};
    bool tiled[W_COUNT]{};
    __half *w[W_COUNT]{};
    // int8 weight variant (wbits == 8): the tiled matrices as int8 tiles
    // [layer][row tile][k-block][128][64] and fp16 row scales [layer][tiles * 128]
    int wbits = 16;
    int8_t *w8[W_COUNT]{};
    __half *wsc[W_COUNT]{};
    std::vector<uint8_t> wset;  // [W_COUNT][L] (globals use index 0)
    size_t n_missing = 0;

    // slot pool
    float *wkv = nullptr, *shift_att = nullptr, *shift_ffn = nullptr, *occ = nullptr;
    SampleParamsDev *params = nullptr;
    unsigned long long *ndraw = nullptr;

    // activations
    __half *xmix[6]{};
    __half *hw = nullptr, *ha = nullptr, *hv = nullptr, *hg = nullptr, *z = nullptr, *xk = nullptr, *h = nullptr,
           *xo = nullptr;
    float *r = nullptr, *k = nullptr, *v = nullptr, *dec = nullptr, *a = nullptr, *vg = nullptr, *g = nullptr,
          *vfirst = nullptr, *x = nullptr, *logits = nullptr, *lpen = nullptr;
    uint32_t *nz = nullptr;
    int32_t *slots = nullptr, *tokens = nullptr, *next = nullptr;
    // split-K partial sums [MAX_SPLIT][bcap][cols] fp32: r, k, v, the LoRA-down
    // outputs (w, a, v, g) and the residual-stream contributions
    float *pr = nullptr, *pk = nullptr, *pv = nullptr, *phw = nullptr, *pha = nullptr, *phv = nullptr,
          *phg = nullptr, *px = nullptr;
    uint32_t *errw = nullptr;
    // per layer: key-projection items stored (fused channel mix); per layer:
    // LoRA-down tiles finished (fused r, k, v + LoRA launch); per layer
    // FIX_TILES_PER_LAYER split-tile counters of that launch; zeroed per step
    uint32_t *ffn_dep = nullptr;
    unsigned long long *nzstat = nullptr;  // nonzero channel-mix blocks counted by the key projection
    unsigned long long nz_considered = 0;  // blocks those counts cover (host side)
    // prefill: second residual buffer and WKV work buffers [bcap][d] ([bcap][H] bonus)
    float *x2 = nullptr, *pf_vec = nullptr, *pf_y = nullptr, *pf_bonus = nullptr;

    CUtensorMap wmap[W_COUNT]{};
    CUtensorMap wmap8[W_COUNT]{};  // int8 tiles, two k-blocks per copy
    CUtensorMap wmap8_1[W_COUNT]{};  // int8 tiles, one k-block per copy
    bool has_wmap[W_COUNT]{};
    CUtensorMap amap[A_COUNT][MAX_B / 16]{};
    bool amap_ok[A_COUNT][MAX_B / 16]{};
    CUtensorMap amap3[A_COUNT][MAX_B / 16]{};  // (col, row, k-block) view: two k-blocks per copy
    bool amap3_ok[A_COUNT][MAX_B / 16]{};
    void *abase[A_COUNT]{};
    int acols[A_COUNT]{};

    std::map<std::tuple<int, int, int, int, int>, cudaGraphExec_t> graphs;
    // in-graph timeline (rwkv7_step_timeline): four words per launch, and the
    // kernel class of each launch of the captured step
    unsigned long long *tlbuf = nullptr;
    std::map<std::tuple<int, int, int>, std::vector<int>> tl_classes;
    std::vector<void *> allocs;
    DevAllocator alloc;  // the allocator in effect when the ctx was created
    Prof prof;
};

namespace {

int fail(rwkv7_ctx *c, int code, const char *fmt, ...) {
    if (c) {
        char buf[512];
        va_list ap;
        va_start(ap, fmt);
        vsnprintf(buf, sizeof buf, fmt, ap);
        va_end(ap);
        c->err = buf;
    }
    return code;
}

#define CK(call)                                                                                   \
    do {                                                                                           \
        cudaError_t e_ = (call);                                                                   \
        if (e_ != cudaSuccess) return fail(c, RWKV7_ECUDA, "%s: %s", #call, cudaGetErrorString(e_)); \
    } while (0)

template <typename T>
int dalloc(rwkv7_ctx *c, T **p, size_t count) {
    void *q = nullptr;
    const size_t bytes = count * sizeof(T) + 256;
    if (c->alloc.alloc) {
        if (c->alloc.alloc(c->alloc.user, bytes, &q) != 0 || !q)
            return fail(c, RWKV7_ENOMEM, "the caller's device allocator refused %zu bytes", bytes);
        if ((uintptr_t)q & 255u) {
            c->alloc.release(c->alloc.user, q);
            return fail(c, RWKV7_EINVAL, "the caller's device allocator returned a pointer not 256-byte aligned");
        }
    } else {
        cudaError_t e = cudaMalloc(&q, bytes);
        if (e != cudaSuccess)
            return fail(c, RWKV7_ENOMEM, "cudaMalloc(%zu bytes): %s", count * sizeof(T), cudaGetErrorString(e));
    }
    c->allocs.push_back(q);
    cudaError_t e = cudaMemset(q, 0, bytes);
    if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "cudaMemset: %s", cudaGetErrorString(e));
    *p = (T *)q;
    return RWKV7_OK;
}

bool per_layer(int kind) { return kind >= FIRST_LAYER_KIND; }

int env_int(const char *name, int dflt) {
    const char *v = getenv(name);
    return (v && *v) ? atoi(v) : dflt;
}

int make_map(rwkv7_ctx *c, CUtensorMap *m, void *base, int rank, const uint64_t *dims, const uint64_t *strides_bytes,
             const uint32_t *box, bool int8 = false) {
    auto fn = encode_fn();
    if (!fn) return fail(c, RWKV7_ECUDA, "cuTensorMapEncodeTiled is not available");
    cuuint64_t gd[3], gs[2];
    cuuint32_t bx[3], es[3] = {1, 1, 1};
    for (int i = 0; i < rank; ++i) {
        gd[i] = dims[i];
        bx[i] = box[i];
    }
    for (int i = 0; i < rank - 1; ++i) gs[i] = strides_bytes[i];
    // fp16 tiles land in the SW128 K-major layout the tensor cores read; int8
    // tiles (64-byte rows) land with the 64-byte swizzle and are widened by the
    // kernel
    CUresult r = fn(m, int8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, (cuuint32_t)rank,
                    base, gd, gs, bx, es, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    int8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return fail(c, RWKV7_ECUDA, "cuTensorMapEncodeTiled failed (%d)", (int)r);
    return RWKV7_OK;
}

int row_tiles(const rwkv7_ctx *c, int kind) { return (c->wrows[kind] + GEMM_TILE_M - 1) / GEMM_TILE_M; }
// k-blocks of 64, padded to an even count (the GEMM moves two per pipeline stage)
int kblocks(const rwkv7_ctx *c, int kind) { return ((c->wcols[kind] + GEMM_TILE_K - 1) / GEMM_TILE_K + 1) & ~1; }
size_t layer_elems(const rwkv7_ctx *c, int kind) {
    return c->tiled[kind] ? (size_t)row_tiles(c, kind) * kblocks(c, kind) * GEMM_TILE_M * GEMM_TILE_K
                          : (size_t)c->wrows[kind] * c->wcols[kind];
}

// Weight map over the tile-major layout: 3D {64 k, 128 rows, all tiles of all
// layers}, box {64, 128, 2}: every load is two adjacent k-block tiles, 32 KB
// contiguous.
int make_wmap(rwkv7_ctx *c, int kind) {
    const int layers = per_layer(kind) ? c->L : 1;
    const uint64_t ntiles = (uint64_t)layers * row_tiles(c, kind) * kblocks(c, kind);
    if (c->wbits == 8) {  // 8 KB int8 tiles, 64-byte rows
        uint64_t dims8[3] = {(uint64_t)GEMM_TILE_K, (uint64_t)GEMM_TILE_M, ntiles};
        uint64_t strides8[2] = {(uint64_t)GEMM_TILE_K, (uint64_t)GEMM_TILE_K * GEMM_TILE_M};
        uint32_t box2[3] = {64, 128, 2}, box1[3] = {64, 128, 1};
        c->has_wmap[kind] = true;
        int rc = make_map(c, &c->wmap8[kind], c->w8[kind], 3, dims8, strides8, box2, true);
        if (rc) return rc;
        return make_map(c, &c->wmap8_1[kind], c->w8[kind], 3, dims8, strides8, box1, true);
    }
    uint64_t dims[3] = {(uint64_t)GEMM_TILE_K, (uint64_t)GEMM_TILE_M, ntiles};
    uint64_t strides[2] = {(uint64_t)GEMM_TILE_K * 2, (uint64_t)GEMM_TILE_K * GEMM_TILE_M * 2};
    uint32_t box[3] = {64, 128, 2};
    c->has_wmap[kind] = true;
    return make_map(c, &c->wmap[kind], c->w[kind], 3, dims, strides, box);
}

// Split factor of a launch whose segments hold `tiles` row tiles in all, each
// `pairs` k-block pairs long: enough k-splits that every SM gets about one
// item.  (Finer splits that balance several items per CTA measured slower: each
// split adds a partial slab that the consumer reads.)  Depends only on the
// shapes, so a slot's result does not depend on B.
int split_for(const rwkv7_ctx *c, int tiles, int pairs) {
    const int per_sm = std::max(1, std::min(4, env_int("RWKV7_GEMM_CTAS_PER_SM", 1)));
    const int s = c->nsm * per_sm / std::max(1, tiles);
    return std::max(1, std::min(s, std::min(MAX_SPLIT, pairs)));
}

// Split-tile counters per layer of the fused r, k, v + LoRA launch (LoRA-down
// row tiles of all four LoRAs).
constexpr int FIX_TILES_PER_LAYER = 16;

// Split factor of the LoRA-down items in the fused r, k, v + LoRA launch.
// Unsplit when a LoRA-down tile is no longer than an r, k, v item (s1
// splits); otherwise split to about half an r, k, v item, so that the LoRA
// chain (down, finish, up) ends while r, k, v still stream -- the finish costs
// a few L2 round trips, which pay only against a long chain.  Depends only on
// the shapes.  RWKV7_LORA_SPLIT overrides it (tuning knob).
int lora_split(const rwkv7_ctx *c, int s1) {
    const int pairs = kblocks(c, L_W1) / 2;
    const int item = std::max(1, kblocks(c, L_WR) / 2 / std::max(1, s1));
    int sd = pairs <= item ? 1 : (2 * pairs + item - 1) / item;
    sd = env_int("RWKV7_LORA_SPLIT", sd);
    return std::max(1, std::min(sd, std::min(MAX_SPLIT, pairs)));
}

// Split factors of the step's split-K projections: r, k, v + LoRA-down (s1),
// output (s3) and channel-mix value (s5).
void step_splits(const rwkv7_ctx *c, int *s1, int *s3, int *s5) {
    *s1 = split_for(c, 3 * row_tiles(c, L_WR) + row_tiles(c, L_W1) + row_tiles(c, L_A1) + row_tiles(c, L_V1) +
                           row_tiles(c, L_G1),
                    kblocks(c, L_WR) / 2);
    *s3 = split_for(c, row_tiles(c, L_WO), kblocks(c, L_WO) / 2);
    *s5 = split_for(c, row_tiles(c, L_FV), kblocks(c, L_FV) / 2);
}

// Activation map: 2D {cols (K), bcap rows}, box {64, npad}: one copy per
// k-block brings every slot row of the step.  Encoded lazily per npad.
int make_amap(rwkv7_ctx *c, int which, void *base, int cols) {
    c->abase[which] = base;
    c->acols[which] = cols;
    return RWKV7_OK;
}
// Activation map as a 3D view {64 cols, bcap rows, K/64 k-blocks} (row stride
// K * 2 bytes, k-block stride 128 bytes), box {64, npad, 2}: one copy brings the
// two k-blocks of a pipeline stage in the same shared-memory layout as two 2D
// boxes.  Only for K a multiple of 128, so that no box reaches past a row.
const CUtensorMap *get_amap3(rwkv7_ctx *c, int which, int npad) {
    if (c->acols[which] % 128 != 0) return nullptr;
    CUtensorMap &m = c->amap3[which][npad / 16 - 1];
    if (!c->amap3_ok[which][npad / 16 - 1]) {
        const uint64_t K = (uint64_t)c->acols[which];
        uint64_t dims[3] = {64, (uint64_t)c->bcap, K / 64};
        uint64_t strides[2] = {K * 2, 128};
        uint32_t box[3] = {64, (uint32_t)npad, 2};
        if (make_map(c, &m, c->abase[which], 3, dims, strides, box) != RWKV7_OK) return nullptr;
        c->amap3_ok[which][npad / 16 - 1] = true;
    }
    return &m;
}

const CUtensorMap *get_amap(rwkv7_ctx *c, int which, int npad) {
    CUtensorMap &m = c->amap[which][npad / 16 - 1];
    if (!c->amap_ok[which][npad / 16 - 1]) {
        uint64_t dims[2] = {(uint64_t)c->acols[which], (uint64_t)c->bcap};
        uint64_t strides[1] = {(uint64_t)c->acols[which] * 2};
        uint32_t box[2] = {64, (uint32_t)npad};
        if (make_map(c, &m, c->abase[which], 2, dims, strides, box) != RWKV7_OK) return nullptr;
        c->amap_ok[which][npad / 16 - 1] = true;
    }
    return &m;
}

// ---------------------------------------------------------------- GEMM launches
struct Seg {
    int wkind;    // weight kind
    int xbuf;     // activation buffer
    const __half *xptr;
    int K;
    int epi;
    void *out;
    int ldo;
    const __half *bias;
    int S;        // k-splits (S > 1: raw fp32 partials, slab stride bcap * ldo)
    void *fix_out = nullptr;  // S > 1 in a two-phase launch: the tile's last split finishes it here
    int fix_epi = 0;          // with this fp16 kind
};

// The channel mix runs as one two-phase launch (key projection, then the value
// projection on every SM once all of h is stored) in the fp16 tensor-core
// modes; otherwise as two launches.
bool ffn_fused(const rwkv7_ctx *c, int mode) {
    return c->wbits == 16 && (mode == 0 || mode == 1) && env_int("RWKV7_FUSE_FFN", 1) != 0;  // tuning knob
}

int lora_split(const rwkv7_ctx *c, int s1);
void step_splits(const rwkv7_ctx *c, int *s1, int *s3, int *s5);

// The r, k, v projections, the LoRA down projections and the LoRA up
// projections with their gates run as one two-phase launch: the LoRA-down
// items are phase 0 and counted per finished row tile; the r, k, v items run
// beside them; the LoRA-up items are phase 1 and read the hidden once every
// LoRA-down tile is finished.  The LoRA chain then overlaps the r, k, v weight
// stream instead of following it as two more launches.  fp16 tensor-core
// modes only; with split LoRA-down tiles only while the batch leaves half the
// SMs free of the preceding LayerNorm rows (wider batches measured faster as
// three launches).  Either way the arithmetic is the same, so a slot's result
// does not depend on which path its step took.
bool att_fused(const rwkv7_ctx *c, int mode, int B) {
    if (c->wbits != 16 || (mode != 0 && mode != 1) || env_int("RWKV7_FUSE_ATT", 1) == 0) return false;  // knob
    int s1, s3, s5;
    step_splits(c, &s1, &s3, &s5);
    return lora_split(c, s1) == 1 || 2 * B <= c->nsm;
}

// nseg0 > 0: a two-phase launch whose first nseg0 segments are phase 0 and
// whose phase-1 activations wait, through the counter *dep, for the items of
// the first nsegdep of them (all nseg0 when nsegdep < 0); fp16 tensor-core
// kernel only.  full_grid: one CTA on every SM (else as many as the larger
// phase has items).
int run_gemm(rwkv7_ctx *c, int layer, const Seg *segs, int n, int B, uint32_t *nz_out, const uint32_t *nz_skip,
             const LaunchCfg &lc, int mode, unsigned long long *tl = nullptr, int nseg0 = 0,
             uint32_t *dep = nullptr, int nsegdep = -1, bool full_grid = false, uint32_t *tile_ctr = nullptr) {
    if (nsegdep < 0 || nsegdep > nseg0) nsegdep = nseg0;
    int nfix_tiles = 0;   // tile counters handed out so far
    bool split_dep = false;
    GemmParams p;
    memset(&p, 0, sizeof p);
    p.tl = tl;
    p.skip_seg = n - 1;
    p.nz_count = nz_out ? c->nzstat : nullptr;
    int nmaps = 0;
    int wslot[W_COUNT], aslot[A_COUNT];
    bool x3slot[A_COUNT] = {};
    for (int i = 0; i < W_COUNT; ++i) wslot[i] = -1;
    for (int i = 0; i < A_COUNT; ++i) aslot[i] = -1;
    int item = 0, blk = 0;
    const bool w8 = c->wbits == 8;
    // int8 weights: k-blocks per ring stage -- pairs while the activation boxes
    // are small, single k-blocks for wide batches (so that four stages fit)
    const int kbs8 = (B + 15) / 16 * 16 > 128 ? 1 : 2;
    for (int s = 0; s < n; ++s) {
        const Seg &sg = segs[s];
        GemmSeg &g = p.seg[s];
        const int rows = c->wrows[sg.wkind];
        if (!c->tiled[sg.wkind] || sg.K != c->wcols[sg.wkind] || sg.S < 1 || sg.S > MAX_SPLIT)
            return fail(c, RWKV7_ECUDA, "internal: bad GEMM segment");
        if (wslot[sg.wkind] < 0) {
            if (nmaps >= GEMM_MAX_MAPS) return fail(c, RWKV7_ECUDA, "too many tensor maps in one GEMM");
            wslot[sg.wkind] = nmaps;
            p.maps[nmaps++] = w8 ? (kbs8 == 2 ? c->wmap8[sg.wkind] : c->wmap8_1[sg.wkind]) : c->wmap[sg.wkind];
        }
        if (aslot[sg.xbuf] < 0) {
            if (nmaps >= GEMM_MAX_MAPS) return fail(c, RWKV7_ECUDA, "too many tensor maps in one GEMM");
            const int np16 = (B + 15) / 16 * 16;
            const CUtensorMap *am3 = (!w8 || kbs8 == 2) ? get_amap3(c, sg.xbuf, np16) : nullptr;
            const CUtensorMap *am = am3 ? am3 : get_amap(c, sg.xbuf, np16);
            if (!am) return RWKV7_ECUDA;
            aslot[sg.xbuf] = nmaps;
            x3slot[sg.xbuf] = am3 != nullptr;
            p.maps[nmaps++] = *am;
        }
        g.wmap = wslot[sg.wkind];
        g.xmap = aslot[sg.xbuf];
        g.x3 = x3slot[sg.xbuf] ? 1 : 0;
        g.rows = rows;
        g.K = sg.K;
        g.kb = kblocks(c, sg.wkind);
        g.tiles = row_tiles(c, sg.wkind);
        g.S = std::min(sg.S, g.kb / 2);
        g.tile_base = (per_layer(sg.wkind) ? layer : 0) * g.tiles * g.kb;
        g.epi = sg.epi;
        g.out = sg.out;
        g.ldo = sg.ldo;
        g.split_stride = (long long)c->bcap * sg.ldo;
        g.bias = sg.bias;
        g.w = w8 ? nullptr : c->w[sg.wkind] + (size_t)(per_layer(sg.wkind) ? layer : 0) * layer_elems(c, sg.wkind);
        g.wscale = w8 ? c->wsc[sg.wkind] + (size_t)(per_layer(sg.wkind) ? layer : 0) * g.tiles * GEMM_TILE_M
                      : nullptr;
        g.x = sg.xptr;
        g.ldx = sg.K;
        if (mode == 2) {
            g.item0 = blk;
            blk += ((rows + 63) / 64) * g.S;
        } else {
            g.item0 = item;
            item += g.tiles * g.S;
        }
        if (sg.fix_out != nullptr) {  // a split finished in the launch (counted per tile)
            if (s >= nsegdep || g.S < 2 || !tile_ctr || nfix_tiles + g.tiles > FIX_TILES_PER_LAYER)
                return fail(c, RWKV7_ECUDA, "internal: bad split fix-up segment");
            g.fix_out = sg.fix_out;
            g.fix_epi = sg.fix_epi;
            g.fix_ctr = tile_ctr + nfix_tiles;
            nfix_tiles += g.tiles;
            split_dep = true;
        }
        if (s < nsegdep) p.dep_target += g.fix_out ? g.tiles : g.tiles * g.S;
        if (s + 1 == nseg0) p.n0 = item;  // phase-0 items: those of the first nseg0 segments
        if (s + 1 == nsegdep) p.ndep = item;  // of which those that feed phase 1
    }
    p.nseg = n;
    p.nmaps = nmaps;
    p.nitems = item;
    p.B = B;
    p.npad = (B + 15) / 16 * 16;
    p.nz_out = nz_out;
    p.nz_skip = nz_skip;
    p.err = c->errw;
    cudaError_t e = cudaSuccess;
    if (mode == 2) {
        if (w8) return fail(c, RWKV7_EINVAL, "the CUDA-core GEMM takes fp16 weights only");
        launch_gemm_simt(p, lc, &e);
    } else if (w8) {
        // Shared memory: ring W (int8 tiles, 8 stages: a multiple of four, see
        // gemm_tc8_kernel) and ring X (activations) as deep as the rest allows;
        // tensor memory: the accumulators and four widened weight stages
        // (kbs8 x 32 columns each) in its 512 columns.  One CTA per SM.
        p.kbs = kbs8;
        const int SB = 4, SW = 8;
        p.accbufs = (2 * p.npad + SB * kbs8 * 32 <= 512) ? 2 : 1;
        const size_t wb = (size_t)kbs8 * GEMM_TILE_M * GEMM_TILE_K;
        const size_t xb = (size_t)kbs8 * p.npad * 128;
        const size_t budget = (size_t)gemm_tc_max_smem() - 2048;
        const int SX = (int)std::min<size_t>(8, (budget - SW * wb) / xb);
        if (SX < 2 || p.accbufs * p.npad + SB * kbs8 * 32 > 512)
            return fail(c, RWKV7_ECUDA, "internal: int8 GEMM buffers do not fit");
        p.stages = SW;
        p.stages_b = SB;
        p.stages_x = SX;
        p.prefetch = 0;  // the int8 producer never waits for the predecessor
        const int grid = std::min(p.nitems, c->nsm);
        launch_gemm_tc8(p, grid, gemm_tc8_smem_bytes(p.npad, kbs8, SW, SX), lc, &e);
    } else {
        // CTAs per SM and pipeline depth: by default one CTA per SM with the
        // deepest pipeline that fits; RWKV7_GEMM_CTAS_PER_SM / RWKV7_GEMM_STAGES
        // override them (tuning knobs).
        const size_t stage = gemm_tc_stage_bytes(p.npad);
        const int per_sm = std::max(1, std::min(4, env_int("RWKV7_GEMM_CTAS_PER_SM", 1)));
        const size_t budget = (size_t)gemm_tc_max_smem() / per_sm - (per_sm > 1 ? 8192 : 2048);
        int stages = (int)std::min<size_t>(6, budget / stage);
        stages = std::max(2, std::min(stages, env_int("RWKV7_GEMM_STAGES", stages)));
        p.stages = stages;
        p.kbs = 2;
        // Two accumulators (the next item's MMAs overlap this item's epilogue)
        // when they fit in the 512 TMEM columns; a CTA of this kernel always
        // has its SM to itself (its shared memory is over half of the SM's),
        // so it may take all of them.
        p.accbufs = (2 * p.npad * per_sm <= 512) ? 2 : 1;
        // weights fetched before the dependency wait, except by a launch that
        // skips stages by flags its predecessor writes (in a two-phase launch
        // only the first phase-1 stages are fetched regardless of the flags)
        p.prefetch = (nz_skip == nullptr || nseg0 > 0) ? env_int("RWKV7_PREFETCH_STAGES", stages) : 0;  // knob
        int grid = std::min(p.nitems, c->nsm * per_sm);
        if (nseg0 > 0) {  // every CTA resident at once: one per SM
            if (!dep || mode == 2 || w8) return fail(c, RWKV7_ECUDA, "internal: two-phase launch");
            p.dep = dep;
            p.g0 = std::min(p.n0, c->nsm);
            grid = full_grid ? c->nsm : std::min(c->nsm, std::max(p.g0, p.nitems - p.n0));
            // Phase-1 CTAs.  Where only some phase-0 items feed phase 1 (the
            // chain), phase 1 goes where it starts soonest.  The predecessor
            // (one LayerNorm row per CTA, a whole SM each) holds B SMs when
            // this launch begins, and the CTAs placed there start late, so
            // with split (short) chain items phase 1 runs on the first
            // nsm - B CTAs: the chain's and the early r, k, v ones.  Without
            // such room (B near nsm or more), on the chain's CTAs and the idle
            // ones; with unsplit (long) chain items, on every CTA but the
            // chain's.
            p.p1a = p.p1b = 0;
            if (p.ndep < p.n0) {
                int gdep = 0;  // CTAs holding items of [0, ndep)
                while (gdep < p.g0 && (long long)gdep * p.n0 / p.g0 < p.ndep) ++gdep;
                const int early = c->nsm - B;
                const int n1 = p.nitems - p.n0;
                int pm = !split_dep ? 0 : (early >= gdep + 1 && early >= n1 / 2) ? 3 : 0;
                pm = env_int("RWKV7_PHASE1_CTAS", pm);  // tuning knob
                if (pm == 3) {
                    p.p1a = std::min(early, grid);
                    p.p1b = grid;
                } else if (pm == 1) {
                    p.p1a = gdep;
                    p.p1b = p.g0;
                } else if (pm == 0) {
                    p.p1b = gdep;
                }
            }
            if (p.p1a + grid - p.p1b < 1) return fail(c, RWKV7_ECUDA, "internal: two-phase launch without phase-1 CTAs");
            p.accbufs = (2 * p.npad <= 512) ? 2 : 1;
        }
        launch_gemm_tc(p, grid, gemm_tc_smem_bytes(p.npad, stages), lc, &e);
    }
    if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "GEMM launch: %s", cudaGetErrorString(e));
    return RWKV7_OK;
}

const __half *LW(rwkv7_ctx *c, int kind, int l) { return c->w[kind] + (size_t)l * layer_elems(c, kind); }

constexpr int TL_MAX_LAUNCHES = 4096;

// Enqueue one fused step for rows [0, B) of the activation buffers (slots and
// tokens already in c->slots / c->tokens).  With `tcls`, every launch gets its
// four timeline words in c->tlbuf (in launch order) and its class is appended.
int enqueue_step(rwkv7_ctx *c, cudaStream_t st, int B, bool head, bool sample, int mode, Prof *pf = nullptr,
                 std::vector<int> *tcls = nullptr) {
    LaunchCfg lc{st, mode != 2 && pf == nullptr};
    LaunchCfg lc0{st, false};
    cudaError_t e = cudaSuccess;
    auto tlp = [&](int cls) -> unsigned long long * {
        if (!tcls || (int)tcls->size() >= TL_MAX_LAUNCHES) return nullptr;
        tcls->push_back(cls);
        return c->tlbuf + 4 * (tcls->size() - 1);
    };
    // optional CUDA-event bracketing of every launch (profiling mode only)
    auto pb = [&](int cls) {
        if (!pf) return;
        if (pf->n + 2 > pf->ev.size()) {
            for (int i = 0; i < 64; ++i) {
                cudaEvent_t ev;
                cudaEventCreate(&ev);
                pf->ev.push_back(ev);
            }
        }
        pf->cls.push_back(cls);
        cudaEventRecord(pf->ev[pf->n++], st);
    };
    auto pe = [&]() {
        if (pf) cudaEventRecord(pf->ev[pf->n++], st);
    };
    const int d = c->d;
    ElemParams ep;
    memset(&ep, 0, sizeof ep);
    ep.single_slot = -1;
    ep.B = B;
    ep.d = d;
    ep.H = c->H;
    ep.F = c->F;
    ep.V = c->V;
    ep.n_slots = c->n_slots;
    ep.L = c->L;
    ep.slots = c->slots;
    ep.tokens = c->tokens;
    ep.x = c->x;
    ep.err = c->errw;
    ep.emb = c->w[W_EMB];
    ep.ln_w = c->w[W_LN0W];
    ep.ln_b = c->w[W_LN0B];
    const bool fuse_ffn = ffn_fused(c, mode), fuse_att = att_fused(c, mode, B);
    if (fuse_ffn || fuse_att) {  // the per-layer counters of the two-phase launches start at zero every step
        e = cudaMemsetAsync(c->ffn_dep, 0, (2 + FIX_TILES_PER_LAYER) * (size_t)c->L * 4, st);
        if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "counter reset: %s", cudaGetErrorString(e));
    }
    pb(P_EMBED);
    ep.tl = tlp(P_EMBED);
    launch_embed(ep, lc0, &e);
    ep.tl = nullptr;
    pe();
    if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "embed launch: %s", cudaGetErrorString(e));
    int rc;
    int s1, s3, s5;  // depend only on the shapes, so a slot's result does not depend on B
    step_splits(c, &s1, &s3, &s5);
    const int sd = lora_split(c, s1);
    const long long xstride = (long long)c->bcap * d;
    int px_splits = 0;  // residual partial slabs in c->px still to be added to x
    for (int l = 0; l < c->L; ++l) {
        // (x += pending partials) + LN1 + token shift + 6 mixes
        ElemParams m = ep;
        m.layer = l;
        m.ln_w = LW(c, L_LN1W, l);
        m.ln_b = LW(c, L_LN1B, l);
        const int mk[6] = {L_XR, L_XW, L_XK, L_XV, L_XA, L_XG};
        for (int q = 0; q < 6; ++q) {
            m.mu[q] = LW(c, mk[q], l);
            m.xo[q] = c->xmix[q];
        }
        m.shift = c->shift_att + (size_t)l * c->n_slots * d;
        m.part = px_splits ? c->px : nullptr;
        m.nsplit = px_splits;
        m.split_stride = xstride;
        pb(P_LN_MIX);
        m.tl = tlp(P_LN_MIX);
        launch_ln_mix(m, 6, lc, &e);
        pe();
        if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "ln_mix launch: %s", cudaGetErrorString(e));
        // LoRA up projections with their gates (G2)
        Seg g2[4];
        int n2 = 0;
        g2[n2++] = {L_W2, A_HW, c->hw, c->rw, EPI_DECAY, c->dec, d, LW(c, L_W0, l), 1};
        g2[n2++] = {L_A2, A_HA, c->ha, c->ra, EPI_SIGMOID_BIAS, c->a, d, LW(c, L_A0, l), 1};
        if (l > 0) g2[n2++] = {L_V2, A_HV, c->hv, c->rv, EPI_SIGMOID_BIAS, c->vg, d, LW(c, L_V0, l), 1};
        g2[n2++] = {L_G2, A_HG, c->hg, c->rg, EPI_F32, c->g, d, nullptr, 1};
        if (fuse_att) {
            // One two-phase launch: LoRA down (unsplit, activated fp16 hidden;
            // counted), r, k, v (s1 partial slabs, beside the chain), then the
            // LoRA up projections (phase 1).
            Seg ga[11];
            int na = 0;
            if (sd == 1) {
                ga[na++] = {L_W1, A_XW, c->xmix[1], d, EPI_F16_TANH, c->hw, c->rw, nullptr, 1};
                ga[na++] = {L_A1, A_XA, c->xmix[4], d, EPI_F16, c->ha, c->ra, nullptr, 1};
                if (l > 0) ga[na++] = {L_V1, A_XV, c->xmix[3], d, EPI_F16, c->hv, c->rv, nullptr, 1};
                ga[na++] = {L_G1, A_XG, c->xmix[5], d, EPI_F16_SIGMOID, c->hg, c->rg, nullptr, 1};
            } else {  // sd partial slabs per tile, finished by the tile's last split
                ga[na++] = {L_W1, A_XW, c->xmix[1], d, EPI_F32, c->phw, c->rw, nullptr, sd, c->hw, EPI_F16_TANH};
                ga[na++] = {L_A1, A_XA, c->xmix[4], d, EPI_F32, c->pha, c->ra, nullptr, sd, c->ha, EPI_F16};
                if (l > 0) ga[na++] = {L_V1, A_XV, c->xmix[3], d, EPI_F32, c->phv, c->rv, nullptr, sd, c->hv, EPI_F16};
                ga[na++] = {L_G1, A_XG, c->xmix[5], d, EPI_F32, c->phg, c->rg, nullptr, sd, c->hg, EPI_F16_SIGMOID};
            }
            const int ndown = na;
            ga[na++] = {L_WR, A_XR, c->xmix[0], d, EPI_F32, c->pr, d, nullptr, s1};
            ga[na++] = {L_WK, A_XK, c->xmix[2], d, EPI_F32, c->pk, d, nullptr, s1};
            ga[na++] = {L_WV, A_XV, c->xmix[3], d, EPI_F32, c->pv, d, nullptr, s1};
            const int nph0 = na;
            for (int q = 0; q < n2; ++q) ga[na++] = g2[q];
            pb(P_GEMM_PROJ);
            if ((rc = run_gemm(c, l, ga, na, B, nullptr, nullptr, lc, mode, tlp(P_GEMM_PROJ), nph0,
                               c->ffn_dep + c->L + l, ndown, true, c->ffn_dep + 2 * (size_t)c->L + (size_t)FIX_TILES_PER_LAYER * l)))
                return rc;
            pe();
        } else {
        // G1: r, k, v as s1 partial slabs and the LoRA down projections as sd
        // (the fused launch's split).  Without a LoRA-down split the epilogues
        // apply the activation and write the fp16 hidden themselves (the LoRA
        // finalize kernel would only convert).
        const bool fin_fused = sd == 1;
        Seg g1[7];
        int n1 = 0;
        g1[n1++] = {L_WR, A_XR, c->xmix[0], d, EPI_F32, c->pr, d, nullptr, s1};
        g1[n1++] = {L_WK, A_XK, c->xmix[2], d, EPI_F32, c->pk, d, nullptr, s1};
        g1[n1++] = {L_WV, A_XV, c->xmix[3], d, EPI_F32, c->pv, d, nullptr, s1};
        if (fin_fused) {
            g1[n1++] = {L_W1, A_XW, c->xmix[1], d, EPI_F16_TANH, c->hw, c->rw, nullptr, 1};
            g1[n1++] = {L_A1, A_XA, c->xmix[4], d, EPI_F16, c->ha, c->ra, nullptr, 1};
            if (l > 0) g1[n1++] = {L_V1, A_XV, c->xmix[3], d, EPI_F16, c->hv, c->rv, nullptr, 1};
            g1[n1++] = {L_G1, A_XG, c->xmix[5], d, EPI_F16_SIGMOID, c->hg, c->rg, nullptr, 1};
        } else {
            g1[n1++] = {L_W1, A_XW, c->xmix[1], d, EPI_F32, c->phw, c->rw, nullptr, sd};
            g1[n1++] = {L_A1, A_XA, c->xmix[4], d, EPI_F32, c->pha, c->ra, nullptr, sd};
            if (l > 0) g1[n1++] = {L_V1, A_XV, c->xmix[3], d, EPI_F32, c->phv, c->rv, nullptr, sd};
            g1[n1++] = {L_G1, A_XG, c->xmix[5], d, EPI_F32, c->phg, c->rg, nullptr, sd};
        }
        pb(P_GEMM_PROJ);
        if ((rc = run_gemm(c, l, g1, n1, B, nullptr, nullptr, lc, mode, tlp(P_GEMM_PROJ)))) return rc;
        pe();
        // LoRA down: add the slabs, activation, fp16 (the LoRA-up GEMM's operands)
        if (!fin_fused) {
        LoraFinParams lf;
        memset(&lf, 0, sizeof lf);
        lf.B = B;
        lf.S = sd;
        lf.r[0] = c->rw; lf.r[1] = c->ra; lf.r[2] = l > 0 ? c->rv : 0; lf.r[3] = c->rg;
        lf.part[0] = c->phw; lf.part[1] = c->pha; lf.part[2] = c->phv; lf.part[3] = c->phg;
        lf.out[0] = c->hw; lf.out[1] = c->ha; lf.out[2] = c->hv; lf.out[3] = c->hg;
        lf.act[0] = 1; lf.act[1] = 0; lf.act[2] = 0; lf.act[3] = 2;
        lf.bcap = c->bcap;
        pb(P_LORA_FIN);
        lf.tl = tlp(P_LORA_FIN);
        launch_lora_fin(lf, lc, &e);
        pe();
        if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "lora_fin launch: %s", cudaGetErrorString(e));
        }
        pb(P_GEMM_LORA);
        if ((rc = run_gemm(c, l, g2, n2, B, nullptr, nullptr, lc, mode, tlp(P_GEMM_LORA)))) return rc;
        pe();
        }
        // WKV7 + GroupNorm + bonus + gate (adds the r, k, v slabs)
        WkvParams wp;
        memset(&wp, 0, sizeof wp);
        wp.B = B;
        wp.d = d;
        wp.H = c->H;
        wp.n_slots = c->n_slots;
        wp.layer = l;
        wp.slots = c->slots;
        wp.r = c->pr;
        wp.k = c->pk;
        wp.v = c->pv;
        wp.nsplit = s1;
        wp.split_stride = xstride;
        wp.dec = c->dec;
        wp.a = c->a;
        wp.vg = c->vg;
        wp.g = c->g;
        wp.v_first = c->vfirst;
        wp.k_k = LW(c, L_KK, l);
        wp.k_a = LW(c, L_KA, l);
        wp.r_k = LW(c, L_RK, l);
        wp.lnx_w = LW(c, L_LNXW, l);
        wp.lnx_b = LW(c, L_LNXB, l);
        wp.wkv = c->wkv + (size_t)l * c->n_slots * c->H * HS * HS;
        wp.z = c->z;
        wp.err = c->errw;
        pb(P_WKV);
        wp.tl = tlp(P_WKV);
        launch_wkv(wp, lc, &e);
        pe();
        if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "wkv launch: %s", cudaGetErrorString(e));
        // G3: output projection, as residual partial slabs
        Seg g3[1] = {{L_WO, A_Z, c->z, d, EPI_F32, c->px, d, nullptr, s3}};
        pb(P_GEMM_OUT);
        if ((rc = run_gemm(c, l, g3, 1, B, nullptr, nullptr, lc, mode, tlp(P_GEMM_OUT)))) return rc;
        pe();
        px_splits = s3;
        // (x += slabs) + LN2 + token shift + mix
        ElemParams m2 = ep;
        m2.layer = l;
        m2.ln_w = LW(c, L_LN2W, l);
        m2.ln_b = LW(c, L_LN2B, l);
        m2.mu[0] = LW(c, L_FXK, l);
        m2.xo[0] = c->xk;
        m2.shift = c->shift_ffn + (size_t)l * c->n_slots * d;
        m2.part = c->px;
        m2.nsplit = px_splits;
        m2.split_stride = xstride;
        pb(P_LN_MIX);
        m2.tl = tlp(P_LN_MIX);
        launch_ln_mix(m2, 1, lc, &e);
        pe();
        if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "ln_mix launch: %s", cudaGetErrorString(e));
        // G4: key + ReLU^2 (+ nonzero flags per 64 hidden units)
        Seg g4[2] = {{L_FK, A_XKF, c->xk, d, EPI_RELU2, c->h, c->F, nullptr, 1},
                     // G5: value over the nonzero hidden blocks, as residual partial slabs
                     {L_FV, A_H, c->h, c->F, EPI_F32, c->px, d, nullptr, s5}};
        if (fuse_ffn) {
            pb(P_GEMM_FFN);
            if ((rc = run_gemm(c, l, g4, 2, B, c->nz, c->nz, lc, mode, tlp(P_GEMM_FFN), 1, c->ffn_dep + l)))
                return rc;
            pe();
        } else {
            pb(P_GEMM_KEY);
            if ((rc = run_gemm(c, l, g4, 1, B, c->nz, nullptr, lc, mode, tlp(P_GEMM_KEY)))) return rc;
            pe();
            pb(P_GEMM_VALUE);
            if ((rc = run_gemm(c, l, g4 + 1, 1, B, nullptr, c->nz, lc, mode, tlp(P_GEMM_VALUE)))) return rc;
            pe();
        }
        px_splits = s5;
    }
    if (head) {
        ElemParams o = ep;
        o.ln_w = c->w[W_LNOW];
        o.ln_b = c->w[W_LNOB];
        o.xo[0] = c->xo;
        o.part = c->px;
        o.nsplit = px_splits;
        o.split_stride = xstride;
        pb(P_LN_OUT);
        o.tl = tlp(P_LN_OUT);
        launch_ln_out(o, lc, &e);
        pe();
        if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "ln_out launch: %s", cudaGetErrorString(e));
        Seg gh[1] = {{W_HEAD, A_XO, c->xo, d, EPI_F32, c->logits, c->V, nullptr, 1}};
        pb(P_GEMM_HEAD);
        if ((rc = run_gemm(c, 0, gh, 1, B, nullptr, nullptr, lc, mode, tlp(P_GEMM_HEAD)))) return rc;
        pe();
        if (sample) {
            SamplerParams sp;
            memset(&sp, 0, sizeof sp);
            sp.B = B;
            sp.V = c->V;
            sp.n_slots = c->n_slots;
            sp.slots = c->slots;
            sp.logits = c->logits;
            sp.occ = c->occ;
            sp.params = c->params;
            sp.ndraw = c->ndraw;
            sp.lpen = c->lpen;
            sp.next = c->next;
            sp.err = c->errw;
            pb(P_SAMPLER);
            sp.tl = tlp(P_SAMPLER);
            launch_sampler(sp, lc, &e);
            pe();
            if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "sampler launch: %s", cudaGetErrorString(e));
        }
    }
    return RWKV7_OK;
}

// ---------------------------------------------------------------- chunked prefill
// n consecutive tokens of one slot (tokens in c->tokens): the tokens form the
// N side of every projection, so each weight is streamed once per chunk.
int enqueue_prefill(rwkv7_ctx *c, cudaStream_t st, int slot, int n, bool head) {
    const int mode = c->mode;
    LaunchCfg lc{st, mode != 2};
    LaunchCfg lc0{st, false};
    cudaError_t e = cudaSuccess;
    const int d = c->d;
    ElemParams ep;
    memset(&ep, 0, sizeof ep);
    ep.B = n;
    ep.d = d;
    ep.H = c->H;
    ep.F = c->F;
    ep.V = c->V;
    ep.n_slots = c->n_slots;
    ep.L = c->L;
    ep.slots = c->slots;
    ep.tokens = c->tokens;
    ep.x = c->x;
    ep.err = c->errw;
    ep.single_slot = slot;
    ep.emb = c->w[W_EMB];
    ep.ln_w = c->w[W_LN0W];
    ep.ln_b = c->w[W_LN0B];
    launch_embed(ep, lc0, &e);
    if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "embed launch: %s", cudaGetErrorString(e));
    int rc;
    int s1, s3, s5;
    step_splits(c, &s1, &s3, &s5);
    const long long xstride = (long long)c->bcap * d;
    float *xa = c->x, *xb = c->x2;  // residual in, residual out of each LayerNorm phase
    int px_splits = 0;
    for (int l = 0; l < c->L; ++l) {
        ElemParams m = ep;
        m.layer = l;
        m.x = xa;
        m.xout = xb;
        m.ln_w = LW(c, L_LN1W, l);
        m.ln_b = LW(c, L_LN1B, l);
        const int mk[6] = {L_XR, L_XW, L_XK, L_XV, L_XA, L_XG};
        for (int q = 0; q < 6; ++q) {
            m.mu[q] = LW(c, mk[q], l);
            m.xo[q] = c->xmix[q];
        }
        m.shift = c->shift_att + (size_t)l * c->n_slots * d;
        m.part = px_splits ? c->px : nullptr;
        m.nsplit = px_splits;
        m.split_stride = xstride;
        launch_ln_mix_prefill(m, 6, lc, &e);
        if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "ln_mix launch: %s", cudaGetErrorString(e));
        Seg g1[7];
        int n1 = 0;
        g1[n1++] = {L_WR, A_XR, c->xmix[0], d, EPI_F32, c->pr, d, nullptr, s1};
        g1[n1++] = {L_WK, A_XK, c->xmix[2], d, EPI_F32, c->pk, d, nullptr, s1};
        g1[n1++] = {L_WV, A_XV, c->xmix[3], d, EPI_F32, c->pv, d, nullptr, s1};
        g1[n1++] = {L_W1, A_XW, c->xmix[1], d, EPI_F32, c->phw, c->rw, nullptr, s1};
        g1[n1++] = {L_A1, A_XA, c->xmix[4], d, EPI_F32, c->pha, c->ra, nullptr, s1};
        if (l > 0) g1[n1++] = {L_V1, A_XV, c->xmix[3], d, EPI_F32, c->phv, c->rv, nullptr, s1};
        g1[n1++] = {L_G1, A_XG, c->xmix[5], d, EPI_F32, c->phg, c->rg, nullptr, s1};
        if ((rc = run_gemm(c, l, g1, n1, n, nullptr, nullptr, lc, mode))) return rc;
        LoraFinParams lf;
        memset(&lf, 0, sizeof lf);
        lf.B = n;
        lf.S = s1;
        lf.r[0] = c->rw; lf.r[1] = c->ra; lf.r[2] = l > 0 ? c->rv : 0; lf.r[3] = c->rg;
        lf.part[0] = c->phw; lf.part[1] = c->pha; lf.part[2] = c->phv; lf.part[3] = c->phg;
        lf.out[0] = c->hw; lf.out[1] = c->ha; lf.out[2] = c->hv; lf.out[3] = c->hg;
        lf.act[0] = 1; lf.act[1] = 0; lf.act[2] = 0; lf.act[3] = 2;
        lf.bcap = c->bcap;
        launch_lora_fin(lf, lc, &e);
        if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "lora_fin launch: %s", cudaGetErrorString(e));
        Seg g2[4];
        int n2 = 0;
        g2[n2++] = {L_W2, A_HW, c->hw, c->rw, EPI_DECAY, c->dec, d, LW(c, L_W0, l), 1};
        g2[n2++] = {L_A2, A_HA, c->ha, c->ra, EPI_SIGMOID_BIAS, c->a, d, LW(c, L_A0, l), 1};
        if (l > 0) g2[n2++] = {L_V2, A_HV, c->hv, c->rv, EPI_SIGMOID_BIAS, c->vg, d, LW(c, L_V0, l), 1};
        g2[n2++] = {L_G2, A_HG, c->hg, c->rg, EPI_F32, c->g, d, nullptr, 1};
        if ((rc = run_gemm(c, l, g2, n2, n, nullptr, nullptr, lc, mode))) return rc;
        WkvSeqParams wp;
        memset(&wp, 0, sizeof wp);
        wp.n = n;
        wp.d = d;
        wp.H = c->H;
        wp.slot = slot;
        wp.n_slots = c->n_slots;
        wp.layer = l;
        wp.r = c->pr;
        wp.k = c->pk;
        wp.v = c->pv;
        wp.nsplit = s1;
        wp.split_stride = xstride;
        wp.dec = c->dec;
        wp.a = c->a;
        wp.vg = c->vg;
        wp.g = c->g;
        wp.v_first = c->vfirst;
        wp.k_k = LW(c, L_KK, l);
        wp.k_a = LW(c, L_KA, l);
        wp.r_k = LW(c, L_RK, l);
        wp.lnx_w = LW(c, L_LNXW, l);
        wp.lnx_b = LW(c, L_LNXB, l);
        wp.vec = c->pf_vec;
        wp.vec_rows = c->bcap;
        wp.bonus = c->pf_bonus;
        wp.y = c->pf_y;
        wp.wkv = c->wkv + (size_t)l * c->n_slots * c->H * HS * HS;
        wp.z = c->z;
        wp.err = c->errw;
        launch_wkv_prefill(wp, lc, &e);
        if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "wkv prefill launch: %s", cudaGetErrorString(e));
        Seg g3[1] = {{L_WO, A_Z, c->z, d, EPI_F32, c->px, d, nullptr, s3}};
        if ((rc = run_gemm(c, l, g3, 1, n, nullptr, nullptr, lc, mode))) return rc;
        ElemParams m2 = ep;
        m2.layer = l;
        m2.x = xb;
        m2.xout = xa;
        m2.ln_w = LW(c, L_LN2W, l);
        m2.ln_b = LW(c, L_LN2B, l);
        m2.mu[0] = LW(c, L_FXK, l);
        m2.xo[0] = c->xk;
        m2.shift = c->shift_ffn + (size_t)l * c->n_slots * d;
        m2.part = c->px;
        m2.nsplit = s3;
        m2.split_stride = xstride;
        launch_ln_mix_prefill(m2, 1, lc, &e);
        if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "ln_mix launch: %s", cudaGetErrorString(e));
        Seg g4[1] = {{L_FK, A_XKF, c->xk, d, EPI_RELU2, c->h, c->F, nullptr, 1}};
        if ((rc = run_gemm(c, l, g4, 1, n, c->nz, nullptr, lc, mode))) return rc;
        Seg g5[1] = {{L_FV, A_H, c->h, c->F, EPI_F32, c->px, d, nullptr, s5}};
        if ((rc = run_gemm(c, l, g5, 1, n, nullptr, c->nz, lc, mode))) return rc;
        px_splits = s5;
    }
    if (head) {  // logits of the last token only
        ElemParams o = ep;
        o.B = 1;
        o.x = xa + (size_t)(n - 1) * d;
        o.ln_w = c->w[W_LNOW];
        o.ln_b = c->w[W_LNOB];
        o.xo[0] = c->xo;
        o.part = c->px + (size_t)(n - 1) * d;
        o.nsplit = px_splits;
        o.split_stride = xstride;
        launch_ln_out(o, lc, &e);
        if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "ln_out launch: %s", cudaGetErrorString(e));
        Seg gh[1] = {{W_HEAD, A_XO, c->xo, d, EPI_F32, c->logits, c->V, nullptr, 1}};
        if ((rc = run_gemm(c, 0, gh, 1, 1, nullptr, nullptr, lc, mode))) return rc;
    }
    return RWKV7_OK;
}

// The CUDA graph of one fused step (captured on first use per key).  A timeline
// graph is the same step with every launch stamping its words in c->tlbuf.
int step_graph(rwkv7_ctx *c, int B, bool head, bool sample, bool timeline, cudaGraphExec_t *out) {
    auto key = std::make_tuple(B, (int)head, (int)sample, c->mode, (int)timeline);
    auto it = c->graphs.find(key);
    if (it == c->graphs.end()) {
        cudaGraph_t g = nullptr;
        std::vector<int> cls;
        if (!c->cap_stream) CK(cudaStreamCreateWithFlags(&c->cap_stream, cudaStreamNonBlocking));
        CK(cudaStreamBeginCapture(c->cap_stream, cudaStreamCaptureModeThreadLocal));
        int rc = enqueue_step(c, c->cap_stream, B, head, sample, 0, nullptr, timeline ? &cls : nullptr);
        cudaError_t e2 = cudaStreamEndCapture(c->cap_stream, &g);
        if (rc) {
            if (g) cudaGraphDestroy(g);
            return rc;
        }
        if (e2 != cudaSuccess) return fail(c, RWKV7_ECUDA, "graph capture: %s", cudaGetErrorString(e2));
        cudaGraphExec_t ex = nullptr;
        cudaError_t e3 = cudaGraphInstantiate(&ex, g, 0);
        cudaGraphDestroy(g);
        if (e3 != cudaSuccess) return fail(c, RWKV7_ECUDA, "graph instantiate: %s", cudaGetErrorString(e3));
        it = c->graphs.emplace(key, ex).first;
        if (timeline) c->tl_classes[std::make_tuple(B, (int)head, (int)sample)] = cls;
    }
    *out = it->second;
    return RWKV7_OK;
}

int run_step(rwkv7_ctx *c, int B, bool head, bool sample) {
    c->nz_considered += (unsigned long long)c->L * ((c->F + 63) / 64);
    if (c->mode != 0) return enqueue_step(c, c->stream, B, head, sample, c->mode);
    cudaGraphExec_t ex = nullptr;
    int rc = step_graph(c, B, head, sample, false, &ex);
    if (rc) return rc;
    CK(cudaGraphLaunch(ex, c->stream));
    return RWKV7_OK;
}


int check_ready(rwkv7_ctx *c) {
    if (c->n_missing) return fail(c, RWKV7_ESTATE, "%zu weight tensors have not been set", c->n_missing);
    return RWKV7_OK;
}

int parse_name(rwkv7_ctx *c, const char *name, int *kind, int *layer) {
    *layer = 0;
    const char *rest = name;
    if (strncmp(name, "blocks.", 7) == 0) {
        char *end = nullptr;
        long l = strtol(name + 7, &end, 10);
        if (end == name + 7 || *end != '.' || l < 0 || l >= c->L) return -1;
        *layer = (int)l;
        rest = end + 1;
        for (int k = FIRST_LAYER_KIND; k < W_COUNT; ++k)
            if (strcmp(rest, kind_name[k]) == 0) {
                *kind = k;
                return 0;
            }
        return -1;
    }
    for (int k = 0; k < FIRST_LAYER_KIND; ++k)
        if (strcmp(rest, kind_name[k]) == 0) {
            *kind = k;
            return 0;
        }
    return -1;
}

}  // namespace

// ============================================================================
// C ABI
// ============================================================================
extern "C" {

int rwkv7_create(const rwkv7_config *cfg, void *cuda_stream, rwkv7_ctx **out) {
    return rwkv7_create_ex(cfg, 16, cuda_stream, out);
}

int rwkv7_create_ex(const rwkv7_config *cfg, int32_t weight_bits, void *cuda_stream, rwkv7_ctx **out) {
    if (!cfg || !out) return RWKV7_EINVAL;
    *out = nullptr;
    if (weight_bits != 16 && weight_bits != 8) return RWKV7_EINVAL;
    const rwkv7_config &g = *cfg;
    if (g.head_size != HS || g.n_layer < 1 || g.d_model < HS || g.d_model % HS || g.d_model > 8192 ||
        g.d_ffn < 64 || g.d_ffn % 64 || g.vocab < 1 || g.n_slots < 1 || g.n_slots > 65536)
        return RWKV7_EINVAL;
    for (int r : {g.lora_w, g.lora_a, g.lora_v, g.lora_g})
        if (r < 8 || r % 8) return RWKV7_EINVAL;
    if (g.vocab % 8) return RWKV7_EINVAL;
    rwkv7_ctx *c = new rwkv7_ctx();
    {
        std::lock_guard<std::mutex> lk(g_alloc_mu);
        c->alloc = g_alloc;
    }
    c->cfg = g;
    c->wbits = weight_bits;
    c->L = g.n_layer;
    c->d = g.d_model;
    c->H = g.d_model / HS;
    c->F = g.d_ffn;
    c->V = g.vocab;
    c->rw = g.lora_w;
    c->ra = g.lora_a;
    c->rv = g.lora_v;
    c->rg = g.lora_g;
    c->n_slots = g.n_slots;
    // activation rows: a fused decode step of up to 256 slots, or a prefill chunk of 256 tokens
    c->bcap = MAX_B;
    c->stream = (cudaStream_t)cuda_stream;
    int dev = 0;
    int rc = RWKV7_OK;
    auto bad = [&](int code) {
        *out = c;  // keep the ctx so the caller can read the error, then destroy it
        return code;
    };
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&c->nsm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return bad(fail(c, RWKV7_ECUDA, "no CUDA device"));
    const int d = c->d, F = c->F, V = c->V, L = c->L;
    auto shp = [&](int k, int rows, int cols) {
        c->wrows[k] = rows;
        c->wcols[k] = cols;
    };
    shp(W_EMB, V, d); shp(W_HEAD, V, d);
    shp(W_LN0W, 1, d); shp(W_LN0B, 1, d); shp(W_LNOW, 1, d); shp(W_LNOB, 1, d);
    for (int k : {L_LN1W, L_LN1B, L_LN2W, L_LN2B, L_XR, L_XW, L_XK, L_XV, L_XA, L_XG, L_W0, L_A0, L_V0, L_KK, L_KA,
                  L_RK, L_LNXW, L_LNXB, L_FXK})
        shp(k, 1, d);
    shp(L_W1, c->rw, d); shp(L_W2, d, c->rw);
    shp(L_A1, c->ra, d); shp(L_A2, d, c->ra);
    shp(L_V1, c->rv, d); shp(L_V2, d, c->rv);
    shp(L_G1, c->rg, d); shp(L_G2, d, c->rg);
    shp(L_WR, d, d); shp(L_WK, d, d); shp(L_WV, d, d); shp(L_WO, d, d);
    shp(L_FK, F, d); shp(L_FV, d, F);
    c->wset.assign((size_t)W_COUNT * L, 0);
    static const int tc_kinds[] = {L_WR, L_WK, L_WV, L_W1, L_A1, L_V1, L_G1, L_W2, L_A2, L_V2, L_G2, L_WO, L_FK, L_FV, W_HEAD};
    for (int k : tc_kinds) c->tiled[k] = true;
    for (int k = 0; k < W_COUNT; ++k) {
        const size_t layers = per_layer(k) ? L : 1;
        if (c->wbits == 8 && c->tiled[k]) {
            if ((rc = dalloc(c, &c->w8[k], layers * layer_elems(c, k)))) return bad(rc);
            if ((rc = dalloc(c, &c->wsc[k], layers * (size_t)row_tiles(c, k) * GEMM_TILE_M))) return bad(rc);
        } else if ((rc = dalloc(c, &c->w[k], layers * layer_elems(c, k)))) {
            return bad(rc);
        }
        c->n_missing += layers;
    }
    for (int k : tc_kinds)
        if ((rc = make_wmap(c, k))) return bad(rc);
    const size_t ns = c->n_slots;
    if ((rc = dalloc(c, &c->wkv, (size_t)L * ns * c->H * HS * HS))) return bad(rc);
    if ((rc = dalloc(c, &c->shift_att, (size_t)L * ns * d))) return bad(rc);
    if ((rc = dalloc(c, &c->shift_ffn, (size_t)L * ns * d))) return bad(rc);
    if ((rc = dalloc(c, &c->occ, ns * V))) return bad(rc);
    if ((rc = dalloc(c, &c->params, ns))) return bad(rc);
    if ((rc = dalloc(c, &c->ndraw, ns))) return bad(rc);
    {
        std::vector<SampleParamsDev> def(ns);
        for (auto &p : def) {
            p.temperature = 1.0f;
            p.top_p = 0.3f;
            p.top_k = 0;
            p.presence = 0.0f;
            p.frequency = 1.0f;
            p.penalty_decay = 0.996f;
            p.seed = 0;
            p.greedy = 0;
            p.pad = 0;
        }
        if (cudaMemcpy(c->params, def.data(), ns * sizeof(SampleParamsDev), cudaMemcpyHostToDevice) != cudaSuccess)
            return bad(fail(c, RWKV7_ECUDA, "params upload"));
    }
    const size_t R = c->bcap;
    for (int q = 0; q < 6; ++q)
        if ((rc = dalloc(c, &c->xmix[q], R * d))) return bad(rc);
    if ((rc = dalloc(c, &c->hw, R * c->rw)) || (rc = dalloc(c, &c->ha, R * c->ra)) ||
        (rc = dalloc(c, &c->hv, R * c->rv)) || (rc = dalloc(c, &c->hg, R * c->rg)) || (rc = dalloc(c, &c->z, R * d)) ||
        (rc = dalloc(c, &c->xk, R * d)) || (rc = dalloc(c, &c->h, R * F)) || (rc = dalloc(c, &c->xo, R * d)))
        return bad(rc);
    if ((rc = dalloc(c, &c->r, R * d)) || (rc = dalloc(c, &c->k, R * d)) || (rc = dalloc(c, &c->v, R * d)) ||
        (rc = dalloc(c, &c->dec, R * d)) || (rc = dalloc(c, &c->a, R * d)) || (rc = dalloc(c, &c->vg, R * d)) ||
        (rc = dalloc(c, &c->g, R * d)) || (rc = dalloc(c, &c->vfirst, R * d)) || (rc = dalloc(c, &c->x, R * d)) ||
        (rc = dalloc(c, &c->logits, R * V)) || (rc = dalloc(c, &c->lpen, R * V)))
        return bad(rc);
    if ((rc = dalloc(c, &c->nz, (size_t)F / 64 + 64))) return bad(rc);
    if ((rc = dalloc(c, &c->slots, R)) || (rc = dalloc(c, &c->tokens, R)) || (rc = dalloc(c, &c->next, R)))
        return bad(rc);
    const size_t SR = (size_t)MAX_SPLIT * R;
    if ((rc = dalloc(c, &c->pr, SR * d)) || (rc = dalloc(c, &c->pk, SR * d)) || (rc = dalloc(c, &c->pv, SR * d)) ||
        (rc = dalloc(c, &c->px, SR * d)) || (rc = dalloc(c, &c->phw, SR * c->rw)) ||
        (rc = dalloc(c, &c->pha, SR * c->ra)) || (rc = dalloc(c, &c->phv, SR * c->rv)) ||
        (rc = dalloc(c, &c->phg, SR * c->rg)))
        return bad(rc);
    if ((rc = dalloc(c, &c->errw, 16))) return bad(rc);
    if ((rc = dalloc(c, &c->ffn_dep, (2 + FIX_TILES_PER_LAYER) * (size_t)L))) return bad(rc);
    if ((rc = dalloc(c, &c->nzstat, 4))) return bad(rc);
    if ((rc = dalloc(c, &c->x2, R * d)) || (rc = dalloc(c, &c->pf_vec, R * 6 * (size_t)d)) ||
        (rc = dalloc(c, &c->pf_y, R * d)) || (rc = dalloc(c, &c->pf_bonus, R * c->H)))
        return bad(rc);
    const int mk[6] = {A_XR, A_XW, A_XK, A_XV, A_XA, A_XG};
    for (int q = 0; q < 6; ++q)
        if ((rc = make_amap(c, mk[q], c->xmix[q], d))) return bad(rc);
    if ((rc = make_amap(c, A_HW, c->hw, c->rw)) || (rc = make_amap(c, A_HA, c->ha, c->ra)) ||
        (rc = make_amap(c, A_HV, c->hv, c->rv)) || (rc = make_amap(c, A_HG, c->hg, c->rg)) ||
        (rc = make_amap(c, A_Z, c->z, d)) || (rc = make_amap(c, A_XKF, c->xk, d)) ||
        (rc = make_amap(c, A_H, c->h, F)) || (rc = make_amap(c, A_XO, c->xo, d)))
        return bad(rc);
    if (cudaDeviceSynchronize() != cudaSuccess) return bad(fail(c, RWKV7_ECUDA, "device sync after create"));
    *out = c;
    return RWKV7_OK;
}

void rwkv7_destroy(rwkv7_ctx *c) {
    if (!c) return;
    cudaStreamSynchronize(c->stream);
    for (auto &kv : c->graphs) cudaGraphExecDestroy(kv.second);
    for (cudaEvent_t ev : c->prof.ev) cudaEventDestroy(ev);
    if (c->cap_stream) cudaStreamDestroy(c->cap_stream);
    for (void *p : c->allocs) {
        if (c->alloc.release)
            c->alloc.release(c->alloc.user, p);
        else
            cudaFree(p);
    }
    delete c;
}

int rwkv7_set_device_allocator(rwkv7_alloc_fn alloc, rwkv7_free_fn release, void *user) {
    if ((alloc == nullptr) != (release == nullptr)) return RWKV7_EINVAL;
    std::lock_guard<std::mutex> lk(g_alloc_mu);
    g_alloc.alloc = alloc;
    g_alloc.release = release;
    g_alloc.user = user;
    return RWKV7_OK;
}

int rwkv7_debug_latch_error(rwkv7_ctx *c, uint32_t flags) {
    if (!c) return RWKV7_EINVAL;
    if (!c->errw) return fail(c, RWKV7_ESTATE, "context not created");
    // stream-ordered read-modify-write of the error word on the host side of a
    // synchronisation: the word is OR-ed exactly as a kernel would latch it
    CK(cudaStreamSynchronize(c->stream));
    uint32_t w = 0;
    CK(cudaMemcpy(&w, c->errw, 4, cudaMemcpyDeviceToHost));
    w |= flags;
    CK(cudaMemcpy(c->errw, &w, 4, cudaMemcpyHostToDevice));
    return RWKV7_OK;
}

const char *rwkv7_last_error(const rwkv7_ctx *c) { return c ? c->err.c_str() : "null context"; }

int rwkv7_set_weight(rwkv7_ctx *c, const char *name, const void *host_f16, size_t bytes) {
    if (!c) return RWKV7_EINVAL;
    if (!name || !host_f16) return fail(c, RWKV7_EINVAL, "null argument");
    int kind, layer;
    if (parse_name(c, name, &kind, &layer)) return fail(c, RWKV7_ESHAPE, "unknown weight name '%s'", name);
    const size_t n = (size_t)c->wrows[kind] * c->wcols[kind];
    if (c->wbits == 8 && c->tiled[kind])
        return fail(c, RWKV7_ESHAPE, "'%s' is an int8 matrix in this context: use rwkv7_set_weight_i8", name);
    if (bytes != n * 2) return fail(c, RWKV7_ESHAPE, "'%s': %zu bytes given, %zu expected", name, bytes, n * 2);
    if (c->tiled[kind]) {
        // repack [rows][cols] into zero-padded 128 x 64 tiles, tile order (row tile, k-block)
        const int rows = c->wrows[kind], cols = c->wcols[kind], kb = kblocks(c, kind);
        std::vector<__half> t(layer_elems(c, kind), __float2half(0.0f));
        const __half *src = (const __half *)host_f16;
        for (int r = 0; r < rows; ++r)
            for (int k0 = 0; k0 < cols; k0 += GEMM_TILE_K) {
                const int nk = std::min(GEMM_TILE_K, cols - k0);
                __half *dst = t.data() + (((size_t)(r / GEMM_TILE_M) * kb + k0 / GEMM_TILE_K) * GEMM_TILE_M +
                                          (r % GEMM_TILE_M)) * GEMM_TILE_K;
                memcpy(dst, src + (size_t)r * cols + k0, (size_t)nk * sizeof(__half));
            }
        CK(cudaMemcpy(c->w[kind] + (size_t)layer * t.size(), t.data(), t.size() * sizeof(__half),
                      cudaMemcpyHostToDevice));
    } else {
        CK(cudaMemcpy(c->w[kind] + (size_t)layer * n, host_f16, bytes, cudaMemcpyHostToDevice));
    }
    uint8_t &f = c->wset[(size_t)kind * c->L + layer];
    if (!f) {
        f = 1;
        c->n_missing--;
    }
    return RWKV7_OK;
}

int rwkv7_set_weight_i8(rwkv7_ctx *c, const char *name, const int8_t *host_q, size_t q_bytes,
                        const void *host_scale_f16, size_t scale_bytes) {
    if (!c) return RWKV7_EINVAL;
    if (!name || !host_q || !host_scale_f16) return fail(c, RWKV7_EINVAL, "null argument");
    int kind, layer;
    if (parse_name(c, name, &kind, &layer)) return fail(c, RWKV7_ESHAPE, "unknown weight name '%s'", name);
    if (c->wbits != 8 || !c->tiled[kind])
        return fail(c, RWKV7_ESHAPE, "'%s' is not an int8 matrix in this context", name);
    const int rows = c->wrows[kind], cols = c->wcols[kind], kb = kblocks(c, kind), tiles = row_tiles(c, kind);
    if (q_bytes != (size_t)rows * cols || scale_bytes != (size_t)rows * 2)
        return fail(c, RWKV7_ESHAPE, "'%s': %zu + %zu bytes given, %zu + %zu expected", name, q_bytes, scale_bytes,
                    (size_t)rows * cols, (size_t)rows * 2);
    // repack [rows][cols] int8 into zero-padded 128 x 64 tiles, tile order (row tile, k-block)
    std::vector<int8_t> t(layer_elems(c, kind), 0);
    for (int r = 0; r < rows; ++r)
        for (int k0 = 0; k0 < cols; k0 += GEMM_TILE_K) {
            const int nk = std::min(GEMM_TILE_K, cols - k0);
            int8_t *dst = t.data() + (((size_t)(r / GEMM_TILE_M) * kb + k0 / GEMM_TILE_K) * GEMM_TILE_M +
                                      (r % GEMM_TILE_M)) * GEMM_TILE_K;
            memcpy(dst, host_q + (size_t)r * cols + k0, (size_t)nk);
        }
    std::vector<__half> sc((size_t)tiles * GEMM_TILE_M, __float2half(0.0f));
    memcpy(sc.data(), host_scale_f16, (size_t)rows * 2);
    CK(cudaMemcpy(c->w8[kind] + (size_t)layer * t.size(), t.data(), t.size(), cudaMemcpyHostToDevice));
    CK(cudaMemcpy(c->wsc[kind] + (size_t)layer * sc.size(), sc.data(), sc.size() * sizeof(__half),
                  cudaMemcpyHostToDevice));
    uint8_t &f = c->wset[(size_t)kind * c->L + layer];
    if (!f) {
        f = 1;
        c->n_missing--;
    }
    return RWKV7_OK;
}

int32_t rwkv7_weight_bits(const rwkv7_ctx *c) { return c ? c->wbits : 0; }

int rwkv7_load_weights(rwkv7_ctx *c, const char *path) {
    if (!c) return RWKV7_EINVAL;
    if (!path) return fail(c, RWKV7_EINVAL, "null path");
    FILE *fh = fopen(path, "rb");
    if (!fh) return fail(c, RWKV7_EINVAL, "cannot open '%s'", path);
    std::vector<char> head(4096 + 1, 0);
    if (fread(head.data(), 1, 4096, fh) != 4096 || strncmp(head.data(), "RWKV7W01\n", 9) != 0) {
        fclose(fh);
        return fail(c, RWKV7_ESHAPE, "'%s' is not an RWKV7W01 weight file", path);
    }
    const char *p = head.data() + 9;
    int n = atoi(p);
    p = strchr(p, '\n');
    int rc = RWKV7_OK;
    std::vector<uint8_t> buf;
    for (int i = 0; i < n && p && rc == RWKV7_OK; ++i) {
        ++p;
        char name[256], dt[16], shape[64];
        unsigned long long off = 0, nb = 0;
        if (sscanf(p, "%255s %15s %63s %llu %llu", name, dt, shape, &off, &nb) != 5 || strcmp(dt, "f16") != 0) {
            rc = fail(c, RWKV7_ESHAPE, "bad header line %d in '%s'", i, path);
            break;
        }
        buf.resize(nb);
        if (fseek(fh, (long)(4096 + off), SEEK_SET) != 0 || fread(buf.data(), 1, nb, fh) != nb) {
            rc = fail(c, RWKV7_ESHAPE, "short read of '%s' in '%s'", name, path);
            break;
        }
        rc = rwkv7_set_weight(c, name, buf.data(), nb);
        p = strchr(p, '\n');
    }
    fclose(fh);
    return rc;
}

static int slot_op(rwkv7_ctx *c, int op, int a, int b) {
    SlotOpParams p;
    memset(&p, 0, sizeof p);
    p.op = op;
    p.a = a;
    p.b = b;
    p.L = c->L;
    p.n_slots = c->n_slots;
    p.wkv_per_slot = (size_t)c->H * HS * HS;
    p.d = c->d;
    p.V = c->V;
    p.wkv = c->wkv;
    p.shift_att = c->shift_att;
    p.shift_ffn = c->shift_ffn;
    p.occ = c->occ;
    p.ndraw = c->ndraw;
    p.params = c->params;
    cudaError_t e = cudaSuccess;
    launch_slot_op(p, c->stream, &e);
    if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "slot op: %s", cudaGetErrorString(e));
    return RWKV7_OK;
}

#define SLOT_OK(s) ((s) >= 0 && (s) < c->n_slots)

int rwkv7_slot_reset(rwkv7_ctx *c, int32_t slot) {
    if (!c) return RWKV7_EINVAL;
    if (!SLOT_OK(slot)) return fail(c, RWKV7_EINVAL, "slot %d out of range", slot);
    return slot_op(c, 0, slot, slot);
}

int rwkv7_slot_swap(rwkv7_ctx *c, int32_t a, int32_t b) {
    if (!c) return RWKV7_EINVAL;
    if (!SLOT_OK(a) || !SLOT_OK(b)) return fail(c, RWKV7_EINVAL, "slot out of range");
    if (a == b) return RWKV7_OK;
    return slot_op(c, 2, a, b);
}

int rwkv7_slot_copy(rwkv7_ctx *c, int32_t src, int32_t dst) {
    if (!c) return RWKV7_EINVAL;
    if (!SLOT_OK(src) || !SLOT_OK(dst)) return fail(c, RWKV7_EINVAL, "slot out of range");
    if (src == dst) return RWKV7_OK;
    return slot_op(c, 1, src, dst);
}

int rwkv7_slot_set_sampling(rwkv7_ctx *c, int32_t slot, const rwkv7_sampling *sp) {
    if (!c) return RWKV7_EINVAL;
    if (!SLOT_OK(slot) || !sp) return fail(c, RWKV7_EINVAL, "bad slot or null params");
    if (!(sp->top_p >= 0.0f) || sp->top_k < 0 || !(sp->penalty_decay >= 0.0f))
        return fail(c, RWKV7_EINVAL, "invalid sampling parameters");
    SampleParamsDev d;
    d.temperature = sp->temperature;
    d.top_p = sp->top_p;
    d.top_k = sp->top_k;
    d.presence = sp->presence;
    d.frequency = sp->frequency;
    d.penalty_decay = sp->penalty_decay;
    d.seed = sp->seed;
    d.greedy = sp->greedy;
    d.pad = 0;
    CK(cudaMemcpyAsync(c->params + slot, &d, sizeof d, cudaMemcpyHostToDevice, c->stream));
    CK(cudaStreamSynchronize(c->stream));
    return RWKV7_OK;
}

size_t rwkv7_slot_state_bytes(const rwkv7_ctx *c) {
    if (!c) return 0;
    return ((size_t)c->L * c->H * HS * HS + 2 * (size_t)c->L * c->d) * sizeof(float);
}

static int state_xfer(rwkv7_ctx *c, int32_t slot, void *host, size_t bytes, bool to_host) {
    if (!SLOT_OK(slot) || !host) return fail(c, RWKV7_EINVAL, "bad slot or null buffer");
    if (bytes != rwkv7_slot_state_bytes(c)) return fail(c, RWKV7_EINVAL, "state buffer must be %zu bytes", rwkv7_slot_state_bytes(c));
    CK(cudaStreamSynchronize(c->stream));
    const size_t per = (size_t)c->H * HS * HS;
    char *hp = (char *)host;
    for (int l = 0; l < c->L; ++l) {
        float *dp = c->wkv + ((size_t)l * c->n_slots + slot) * per;
        if (to_host)
            CK(cudaMemcpy(hp, dp, per * 4, cudaMemcpyDeviceToHost));
        else
            CK(cudaMemcpy(dp, hp, per * 4, cudaMemcpyHostToDevice));
        hp += per * 4;
    }
    float *bases[2] = {c->shift_att, c->shift_ffn};
    for (float *base : bases)
        for (int l = 0; l < c->L; ++l) {
            float *dp = base + ((size_t)l * c->n_slots + slot) * c->d;
            if (to_host)
                CK(cudaMemcpy(hp, dp, (size_t)c->d * 4, cudaMemcpyDeviceToHost));
            else
                CK(cudaMemcpy(dp, hp, (size_t)c->d * 4, cudaMemcpyHostToDevice));
            hp += (size_t)c->d * 4;
        }
    return RWKV7_OK;
}

int rwkv7_slot_get_state(rwkv7_ctx *c, int32_t slot, void *host_buf, size_t bytes) {
    if (!c) return RWKV7_EINVAL;
    return state_xfer(c, slot, host_buf, bytes, true);
}

int rwkv7_slot_set_state(rwkv7_ctx *c, int32_t slot, const void *host_buf, size_t bytes) {
    if (!c) return RWKV7_EINVAL;
    return state_xfer(c, slot, (void *)host_buf, bytes, false);
}

int rwkv7_prefill_seq(rwkv7_ctx *c, int32_t slot, const int32_t *d_tokens, int32_t T, float *d_logits_out) {
    if (!c) return RWKV7_EINVAL;
    if (!SLOT_OK(slot) || !d_tokens || T <= 0) return fail(c, RWKV7_EINVAL, "bad slot, token pointer or length");
    int rc;
    if ((rc = check_ready(c))) return rc;
    // chunks of up to bcap tokens; every weight is streamed once per chunk
    for (int s0 = 0; s0 < T; s0 += c->bcap) {
        const int n = std::min(c->bcap, T - s0);
        CK(cudaMemcpyAsync(c->tokens, d_tokens + s0, (size_t)n * 4, cudaMemcpyDeviceToDevice, c->stream));
        const bool last = (s0 + n == T) && d_logits_out;
        if ((rc = enqueue_prefill(c, c->stream, slot, n, last))) return rc;
        c->nz_considered += (unsigned long long)c->L * ((c->F + 63) / 64);
    }
    if (d_logits_out)
        CK(cudaMemcpyAsync(d_logits_out, c->logits, (size_t)c->V * 4, cudaMemcpyDeviceToDevice, c->stream));
    return RWKV7_OK;
}

int rwkv7_decode_step(rwkv7_ctx *c, const int32_t *d_slots, const int32_t *d_tokens, int32_t B, float *d_logits_out,
                      int32_t *d_next_out) {
    if (!c) return RWKV7_EINVAL;
    if (!d_slots || !d_tokens || B < 1 || B > c->n_slots)
        return fail(c, RWKV7_EINVAL, "bad decode arguments (B=%d, n_slots=%d)", B, c->n_slots);
    int rc;
    if ((rc = check_ready(c))) return rc;
    const bool head = d_logits_out || d_next_out;
    for (int off = 0; off < B; off += MAX_B) {
        const int bs = std::min(MAX_B, B - off);
        if (d_slots + off != c->slots)
            CK(cudaMemcpyAsync(c->slots, d_slots + off, (size_t)bs * 4, cudaMemcpyDeviceToDevice, c->stream));
        if (d_tokens + off != c->tokens)
            CK(cudaMemcpyAsync(c->tokens, d_tokens + off, (size_t)bs * 4, cudaMemcpyDeviceToDevice, c->stream));
        if ((rc = run_step(c, bs, head, d_next_out != nullptr))) return rc;
        if (d_logits_out && d_logits_out + (size_t)off * c->V != c->logits)
            CK(cudaMemcpyAsync(d_logits_out + (size_t)off * c->V, c->logits, (size_t)bs * c->V * 4,
                               cudaMemcpyDeviceToDevice, c->stream));
        if (d_next_out && d_next_out + off != c->next)
            CK(cudaMemcpyAsync(d_next_out + off, c->next, (size_t)bs * 4, cudaMemcpyDeviceToDevice, c->stream));
    }
    return RWKV7_OK;
}

int rwkv7_decode_step_host(rwkv7_ctx *c, const int32_t *h_slots, const int32_t *h_tokens, int32_t B,
                           float *h_logits_out, int32_t *h_next_out) {
    if (!c) return RWKV7_EINVAL;
    if (!h_slots || !h_tokens || B < 1 || B > c->n_slots) return fail(c, RWKV7_EINVAL, "bad decode arguments");
    std::vector<uint8_t> seen(c->n_slots, 0);
    for (int b = 0; b < B; ++b) {
        if (!SLOT_OK(h_slots[b])) return fail(c, RWKV7_EINVAL, "slot %d out of range", h_slots[b]);
        if (seen[h_slots[b]]++) return fail(c, RWKV7_EINVAL, "slot %d repeated", h_slots[b]);
        if (h_tokens[b] < 0 || h_tokens[b] >= c->V) return fail(c, RWKV7_EINVAL, "token %d out of range", h_tokens[b]);
    }
    int rc;
    if ((rc = check_ready(c))) return rc;
    const bool head = h_logits_out || h_next_out;
    for (int off = 0; off < B; off += MAX_B) {
        const int bs = std::min(MAX_B, B - off);
        CK(cudaMemcpyAsync(c->slots, h_slots + off, (size_t)bs * 4, cudaMemcpyHostToDevice, c->stream));
        CK(cudaMemcpyAsync(c->tokens, h_tokens + off, (size_t)bs * 4, cudaMemcpyHostToDevice, c->stream));
        if ((rc = run_step(c, bs, head, h_next_out != nullptr))) return rc;
        if (h_logits_out)
            CK(cudaMemcpyAsync(h_logits_out + (size_t)off * c->V, c->logits, (size_t)bs * c->V * 4,
                               cudaMemcpyDeviceToHost, c->stream));
        if (h_next_out)
            CK(cudaMemcpyAsync(h_next_out + off, c->next, (size_t)bs * 4, cudaMemcpyDeviceToHost, c->stream));
    }
    CK(cudaStreamSynchronize(c->stream));
    return RWKV7_OK;
}

int rwkv7_sample_batch(rwkv7_ctx *c, const int32_t *d_slots, const float *d_logits, int32_t B, int32_t *d_next_out) {
    if (!c) return RWKV7_EINVAL;
    if (!d_slots || !d_logits || !d_next_out || B < 1 || B > c->n_slots)
        return fail(c, RWKV7_EINVAL, "bad sampling arguments");
    for (int off = 0; off < B; off += c->bcap) {
        const int bs = std::min(c->bcap, B - off);
        SamplerParams sp;
        memset(&sp, 0, sizeof sp);
        sp.B = bs;
        sp.V = c->V;
        sp.n_slots = c->n_slots;
        sp.slots = d_slots + off;
        sp.logits = d_logits + (size_t)off * c->V;
        sp.occ = c->occ;
        sp.params = c->params;
        sp.ndraw = c->ndraw;
        sp.lpen = c->lpen;
        sp.next = d_next_out + off;
        sp.err = c->errw;
        cudaError_t e = cudaSuccess;
        launch_sampler(sp, LaunchCfg{c->stream, false}, &e);
        if (e != cudaSuccess) return fail(c, RWKV7_ECUDA, "sampler launch: %s", cudaGetErrorString(e));
    }
    return RWKV7_OK;
}

int rwkv7_synchronize(rwkv7_ctx *c) {
    if (!c) return RWKV7_EINVAL;
    CK(cudaStreamSynchronize(c->stream));
    uint32_t w = 0;
    CK(cudaMemcpy(&w, c->errw, 4, cudaMemcpyDeviceToHost));
    if (w) {
        CK(cudaMemset(c->errw, 0, 4));
        if (w & ERR_TIMEOUT) return fail(c, RWKV7_ETIMEOUT, "a bounded wait inside a kernel gave up (flags 0x%x)", w);
        return fail(c, RWKV7_EINVAL, "device-side argument error (flags 0x%x: %s%s%s%s)", w,
                    (w & ERR_SLOT) ? "slot out of range " : "", (w & ERR_TOKEN) ? "token out of range " : "",
                    (w & ERR_DUP) ? "repeated slot " : "", (w & ERR_CONFIG) ? "sampler found no token" : "");
    }
    return RWKV7_OK;
}

int rwkv7_set_mode(rwkv7_ctx *c, int32_t mode) {
    if (!c) return RWKV7_EINVAL;
    if (mode < 0 || mode > 2) return fail(c, RWKV7_EINVAL, "mode must be 0, 1 or 2");
    if (c->wbits == 8 && mode >= 2)
        return fail(c, RWKV7_EINVAL, "int8 weights run in modes 0 and 1 (tensor-core kernels) only");
    c->mode = mode;
    return RWKV7_OK;
}

int32_t rwkv7_step_kernel_count(const rwkv7_ctx *c, int32_t B, int32_t with_sampling) {
    if (!c || B < 1) return 0;
    int s1, s3, s5;
    step_splits(c, &s1, &s3, &s5);
    // the LoRA finalize kernel runs only for split LoRA-down tiles; the fused
    // channel mix is one launch; the fused r, k, v + LoRA launch replaces three
    int total = 0;
    for (int b0 = 0; b0 < B; b0 += MAX_B) {
        const int nb = std::min(MAX_B, B - b0);
        const int per_layer = (att_fused(c, c->mode, nb) ? 6 : (lora_split(c, s1) == 1 ? 7 : 8)) +
                              (ffn_fused(c, c->mode) ? 0 : 1);
        total += 1 + per_layer * c->L + 2 + (with_sampling ? 1 : 0);
    }
    return total;
}

int rwkv7_ffn_union_stats(rwkv7_ctx *c, uint64_t *nonzero_blocks, uint64_t *blocks) {
    if (!c) return RWKV7_EINVAL;
    if (!nonzero_blocks || !blocks) return fail(c, RWKV7_EINVAL, "null argument");
    CK(cudaStreamSynchronize(c->stream));
    unsigned long long nz = 0;
    CK(cudaMemcpy(&nz, c->nzstat, sizeof nz, cudaMemcpyDeviceToHost));
    CK(cudaMemset(c->nzstat, 0, sizeof nz));
    *nonzero_blocks = nz;
    *blocks = c->nz_considered;
    c->nz_considered = 0;
    return RWKV7_OK;
}

int rwkv7_profile_step(rwkv7_ctx *c, const int32_t *d_slots, const int32_t *d_tokens, int32_t B,
                       int32_t with_sampling, float *ms_out, int32_t *launches_out, int32_t n_classes) {
    if (!c) return RWKV7_EINVAL;
    if (!d_slots || !d_tokens || !ms_out || !launches_out || B < 1 || B > c->bcap || n_classes < P_COUNT)
        return fail(c, RWKV7_EINVAL, "bad profiling arguments (B must be <= %d, n_classes >= %d)", c->bcap, (int)P_COUNT);
    int rc;
    if ((rc = check_ready(c))) return rc;
    if (d_slots != c->slots) CK(cudaMemcpyAsync(c->slots, d_slots, (size_t)B * 4, cudaMemcpyDeviceToDevice, c->stream));
    if (d_tokens != c->tokens)
        CK(cudaMemcpyAsync(c->tokens, d_tokens, (size_t)B * 4, cudaMemcpyDeviceToDevice, c->stream));
    Prof &pf = c->prof;
    pf.n = 0;
    pf.cls.clear();
    const int mode = c->mode == 2 ? 2 : 1;
    c->nz_considered += (unsigned long long)c->L * ((c->F + 63) / 64);
    if ((rc = enqueue_step(c, c->stream, B, true, with_sampling != 0, mode, &pf))) return rc;
    CK(cudaStreamSynchronize(c->stream));
    for (int i = 0; i < n_classes; ++i) {
        ms_out[i] = 0.0f;
        launches_out[i] = 0;
    }
    for (size_t i = 0; i < pf.cls.size(); ++i) {
        float ms = 0.0f;
        CK(cudaEventElapsedTime(&ms, pf.ev[2 * i], pf.ev[2 * i + 1]));
        ms_out[pf.cls[i]] += ms;
        launches_out[pf.cls[i]] += 1;
    }
    return RWKV7_OK;
}

int rwkv7_step_timeline(rwkv7_ctx *c, const int32_t *d_slots, const int32_t *d_tokens, int32_t B,
                        int32_t with_sampling, uint64_t *host_times, int32_t *host_classes, int32_t max_launches,
                        int32_t *n_launches) {
    if (!c) return RWKV7_EINVAL;
    if (!d_slots || !d_tokens || !host_times || !host_classes || !n_launches || B < 1 || B > c->bcap ||
        max_launches < 1)
        return fail(c, RWKV7_EINVAL, "bad timeline arguments (B must be <= %d)", c->bcap);
    if (c->mode != 0 && c->mode != 1) return fail(c, RWKV7_EINVAL, "the timeline covers modes 0 and 1");
    int rc;
    if ((rc = check_ready(c))) return rc;
    if (!c->tlbuf && (rc = dalloc(c, &c->tlbuf, (size_t)4 * TL_MAX_LAUNCHES))) return rc;
    if (d_slots != c->slots) CK(cudaMemcpyAsync(c->slots, d_slots, (size_t)B * 4, cudaMemcpyDeviceToDevice, c->stream));
    if (d_tokens != c->tokens)
        CK(cudaMemcpyAsync(c->tokens, d_tokens, (size_t)B * 4, cudaMemcpyDeviceToDevice, c->stream));
    // start words to all ones, release-max and end words to zero
    CK(cudaMemsetAsync(c->tlbuf, 0xFF, (size_t)32 * TL_MAX_LAUNCHES, c->stream));
    CK(cudaMemset2DAsync(c->tlbuf + 2, 32, 0, 16, TL_MAX_LAUNCHES, c->stream));
    c->nz_considered += (unsigned long long)c->L * ((c->F + 63) / 64);
    std::vector<int> cls;
    if (c->mode == 0) {
        cudaGraphExec_t ex = nullptr;
        if ((rc = step_graph(c, B, true, with_sampling != 0, true, &ex))) return rc;
        cls = c->tl_classes[std::make_tuple(B, 1, (int)(with_sampling != 0))];
        CK(cudaGraphLaunch(ex, c->stream));
    } else {
        if ((rc = enqueue_step(c, c->stream, B, true, with_sampling != 0, c->mode, nullptr, &cls))) return rc;
    }
    CK(cudaStreamSynchronize(c->stream));
    const int n = std::min((int)cls.size(), (int)max_launches);
    CK(cudaMemcpy(host_times, c->tlbuf, (size_t)n * 32, cudaMemcpyDeviceToHost));
    for (int i = 0; i < n; ++i) host_classes[i] = cls[i];
    *n_launches = n;
    return RWKV7_OK;
}

int rwkv7_get_io_buffers(rwkv7_ctx *c, int32_t **d_slots, int32_t **d_tokens, float **d_logits, int32_t **d_next) {
    if (!c) return RWKV7_EINVAL;
    if (d_slots) *d_slots = c->slots;
    if (d_tokens) *d_tokens = c->tokens;
    if (d_logits) *d_logits = c->logits;
    if (d_next) *d_next = c->next;
    return RWKV7_OK;
}

}  // extern "C"
