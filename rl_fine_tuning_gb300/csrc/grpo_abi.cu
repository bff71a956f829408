// C ABI of libgrpo: argument validation, workspace layout, TMA descriptors and
// the launch sequence of the fused linear GRPO loss.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>
#include <vector>

#include "internal.h"

namespace grpo {

namespace {

constexpr int kVersion = 100;   // 0.1.0

// ---- launch accounting and optional per-kernel event timing
std::atomic<unsigned long long> g_launches{0};

struct ProfRecord {
    int kind;
    cudaEvent_t a, b;
};

// `on` is read by every launch; the records and the event pool are touched
// only while profiling is on, under `mu`.
struct Profiler {
    std::atomic<bool> on{false};
    std::mutex mu;
    std::vector<ProfRecord> recs;
    std::vector<cudaEvent_t> pool;
    cudaEvent_t get() {
        if (!pool.empty()) {
            cudaEvent_t e = pool.back();
            pool.pop_back();
            return e;
        }
        cudaEvent_t e = nullptr;
        if (cudaEventCreate(&e) != cudaSuccess) return nullptr;
        return e;
    }
};
Profiler g_prof;

// launch one kernel through `fn`, counting it and timing it when profiling is on
template <class F>
cudaError_t launch(int kind, cudaStream_t st, F&& fn) {
    if (!g_prof.on.load(std::memory_order_relaxed)) {
        const cudaError_t e = fn();
        if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
        return e;
    }
    std::lock_guard<std::mutex> lock(g_prof.mu);
    cudaEvent_t a = g_prof.get(), b = g_prof.get();
    if (a) cudaEventRecord(a, st);
    const cudaError_t e = fn();
    if (e == cudaSuccess) g_launches.fetch_add(1, std::memory_order_relaxed);
    if (a && b) {
        cudaEventRecord(b, st);
        g_prof.recs.push_back(ProfRecord{kind, a, b});
    }
    return e;
}

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

bool shape_ok(const grpo_shape& s) {
    if (s.n_groups < 1 || s.G < 1 || s.L < 1 || s.V < 1 || s.d < 64 || s.d % 64 != 0) return false;
    if (s.d > 65536 || s.V > (1 << 30)) return false;
    const int64_t N = static_cast<int64_t>(s.n_groups) * s.G * s.L;
    if (N > (1LL << 31) - (1LL << 16)) return false;
    if (s.chunk_rows < 0) return false;
    if (s.loss_mode != GRPO_TOKEN_MEAN && s.loss_mode != GRPO_SEQUENCE_MEAN) return false;
    if (s.objective < GRPO_OBJ_GRPO || s.objective > GRPO_OBJ_FORWARD_KL) return false;
    return true;
}

bool dtype_ok(const grpo_shape& s) { return s.dtype == GRPO_BF16 || s.dtype == GRPO_FP16; }
bool dtype_ok_any(const grpo_shape& s) { return dtype_ok(s) || is_fp8(s.dtype); }

template <class P>
bool aligned(const P* p, size_t a) {
    return (reinterpret_cast<uintptr_t>(p) % a) == 0;
}

struct DeviceInfo {
    int sm_count = 0;
    bool ok = false;
};

int device_info(DeviceInfo* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GRPO_ERR_LAUNCH;
    int major = 0, minor = 0, smc = 0, smem = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smc, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess)
        return GRPO_ERR_LAUNCH;
    if (major != 10 || minor != 3) return GRPO_ERR_DEVICE;
    if (smem < 200 * 1024) return GRPO_ERR_DEVICE;
    out->sm_count = smc;
    out->ok = true;
    return GRPO_OK;
}

// looked up once per process (a thread-safe static initialisation)
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
    static const PFN_cuTensorMapEncodeTiled_v12000 fn = [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            p = nullptr;
        return reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
    }();
    return fn;
}

// 2-D row-major matrix [rows x cols] of 16-bit elements with row pitch `pitch`
// elements, 128-byte swizzled boxes of box_cols x box_rows.
bool make_map(CUtensorMap* m, const void* base, bool bf16, uint64_t cols, uint64_t rows, uint64_t pitch,
              uint32_t box_cols, uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {pitch * 2};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 2,
                    const_cast<void*>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                    CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

// 2-D row-major matrix of 8-bit elements (FP8 codes), 128-byte swizzled boxes
bool make_map_u8(CUtensorMap* m, const void* base, uint64_t cols, uint64_t rows, uint64_t pitch, uint32_t box_cols,
                 uint32_t box_rows) {
    auto fn = encode_fn();
    if (!fn) return false;
    cuuint64_t dims[2] = {cols, rows};
    cuuint64_t strides[1] = {pitch};
    cuuint32_t box[2] = {box_cols, box_rows};
    cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

int default_chunk_rows(const grpo_shape& s) {
    // 8-bit shapes: 76 tiles, so that dW's 8-bit K loop (twice as fast per row as the
    // 16-bit one) stays long against its fp32 read-modify-write epilogue
    if (is_fp8(s.dtype)) return kChunkTilesLarge * kBM;
    const int n_dt = (s.d + kBN - 1) / kBN;
    const int pairs_small = (kChunkTilesSmall + 1) / 2;
    const int tiles = (pairs_small * n_dt) % kChunkPairs == 0 ? kChunkTilesSmall : kChunkTilesLarge;
    return tiles * kBM;
}

int chunk_rows_of(const grpo_shape& s) {
    int r = s.chunk_rows > 0 ? s.chunk_rows : default_chunk_rows(s);
    r = (r + kBM - 1) / kBM * kBM;
    const int64_t N = static_cast<int64_t>(s.n_groups) * s.G * s.L;
    const int64_t nmax = (N + kBM - 1) / kBM * kBM;
    if (r > nmax) r = static_cast<int>(nmax);
    return r;
}

}  // namespace

// splits of n_ntiles vocabulary tiles into at most max_splits ranges, none empty
static void split_vocab(int n_ntiles, int max_splits, int* S, int* nps) {
    int s = n_ntiles < max_splits ? n_ntiles : max_splits;
    *nps = (n_ntiles + s - 1) / s;
    *S = (n_ntiles + *nps - 1) / *nps;
}

// Splits of the chunk forward.  Its static schedule hands every CTA pair the
// same number of (row tile, split) units when a chunk has one row tile per
// pair, so splits of one size give every pair the same work.  Prefer the
// equal division of the vocabulary tiles whose split count is closest to
// `target` within [target/2, max_splits]; without one, fall back to ranges of
// at most `target` splits with a shorter last range.
static void split_vocab_even(int n_ntiles, int target, int max_splits, int* S, int* nps) {
    int best = 0;
    for (int s = target / 2; s <= max_splits && s <= n_ntiles; ++s) {
        if (n_ntiles % s != 0) continue;
        const int dist = s > target ? s - target : target - s;
        const int bdist = best > target ? best - target : target - best;
        if (best == 0 || dist < bdist) best = s;
    }
    if (best == 0) {
        split_vocab(n_ntiles, target, S, nps);
        return;
    }
    *S = best;
    *nps = n_ntiles / best;
}

bool ws_layout(const grpo_shape& s, WsLayout* o) {
    if (!shape_ok(s)) return false;
    const int64_t N = static_cast<int64_t>(s.n_groups) * s.G * s.L;
    o->N = N;
    o->n_ntiles = (s.V + kBN - 1) / kBN;
    split_vocab(o->n_ntiles, kTileSplits, &o->S, &o->nps);
    split_vocab_even(o->n_ntiles, kChunkSplits, kChunkSplitsMax, &o->Sc, &o->npsc);
    o->R = chunk_rows_of(s);
    o->V_pad = (s.V + 63) / 64 * 64;
    o->nc32 = ((s.V + 31) / 32 + 7) / 8 * 8;   // whole 32-byte sectors per 256-column tile
    o->nblk = static_cast<int>((N + kMergeThreads - 1) / kMergeThreads);
    o->n_sched = static_cast<int>(2 + (N + o->R - 1) / o->R);
    o->n_seq = s.n_groups * s.G;
    size_t off = 0;
    auto take = [&](size_t bytes) {
        const size_t at = off;
        off = align_up(off + bytes, 256);
        return at;
    };
    // forward-only path (also what the workspace-free forward uses): everything below `hc`
    o->counts = take(C_COUNT_WORDS * 4);
    o->sched = take(static_cast<size_t>(o->n_sched) * 4);
    o->seqcnt = take(static_cast<size_t>(o->n_seq) * 4);
    o->tiles = take(static_cast<size_t>(N) * 8);
    o->rows = take(static_cast<size_t>(N) * 4);
    o->part = take(static_cast<size_t>(N) * o->S * 16);
    o->zt = take(static_cast<size_t>(N) * 8);
    o->lse = take(static_cast<size_t>(N) * 4);
    o->gco = take(static_cast<size_t>(N) * 4);
    o->ell = take(static_cast<size_t>(N) * 4);
    o->blocksum = take(static_cast<size_t>(o->nblk) * 8);
    // backward chunk buffers
    o->hc = take(static_cast<size_t>(o->R) * s.d * 2);
    o->hcr = take(static_cast<size_t>(o->R) * s.d * 2);
    o->partc = take(static_cast<size_t>(o->R) * o->Sc * 16);
    o->mx = take(static_cast<size_t>(o->R) * o->nc32 * 4);
    o->ds = take(static_cast<size_t>(o->R) * o->V_pad * 2);
    o->hct = take(static_cast<size_t>(o->R) * s.d * 2);
    o->rmax = o->qa = o->qb = o->gmax = o->keys = o->tokpos = 0;
    if (is_fp8(s.dtype)) {
        // the 8-bit backward's buffers (its forward-only entry point needs none of them)
        o->rmax = take(static_cast<size_t>(N) * 4);
        o->qa = take(static_cast<size_t>(o->R) * o->V_pad);
        o->qb = take(static_cast<size_t>(o->R) * o->V_pad);
        o->gmax = take(static_cast<size_t>(o->nc32) * 4);
        o->keys = take(static_cast<size_t>(o->n_sched - 2) * o->R * 8);   // every chunk's keys
        o->tokpos = take(static_cast<size_t>(s.V) * 4);
    }
    o->total = off;
    return true;
}

}  // namespace grpo

using namespace grpo;

namespace {

struct Inputs {
    const void *h_pol, *h_ref, *W;
    const int32_t* tokens;
    const uint8_t* mask;
    const float* adv;
    const grpo_shape* shape;
    void* ws;
    size_t ws_bytes;
    float* loss_out;
    float* row_stats;
    int32_t* status;
    const int32_t* global_counts = nullptr;   // a data-parallel shard: every shard's counts (device [2])
};

int validate(const Inputs& in, WsLayout* L) {
    if (!in.shape) return GRPO_ERR_SHAPE;
    const grpo_shape& s = *in.shape;
    if (!dtype_ok(s)) return GRPO_ERR_DTYPE;
    if (!ws_layout(s, L)) return GRPO_ERR_SHAPE;
    if (!in.h_pol || !in.h_ref || !in.W || !in.tokens || !in.mask || !in.adv || !in.ws || !in.loss_out ||
        !in.status)
        return GRPO_ERR_POINTER;
    if (!aligned(in.h_pol, 16) || !aligned(in.h_ref, 16) || !aligned(in.W, 16) || !aligned(in.tokens, 4) ||
        !aligned(in.adv, 4) || !aligned(in.ws, 256) || !aligned(in.loss_out, 4) || !aligned(in.status, 4) ||
        (in.row_stats && !aligned(in.row_stats, 4)))
        return GRPO_ERR_POINTER;
    if (in.ws_bytes < L->total) return GRPO_ERR_WORKSPACE;
    return GRPO_OK;
}

MergeParams merge_params(const Inputs& in, const WsLayout& L, char* w, int chunk, const float4* part, int S) {
    const grpo_shape& s = *in.shape;
    MergeParams mp;
    mp.part = part;
    mp.zt = reinterpret_cast<const float2*>(w + L.zt);
    mp.mask = in.mask;
    mp.tokens = in.tokens;
    mp.adv = in.adv;
    mp.counts = reinterpret_cast<const int*>(w + L.counts);
    mp.rows = reinterpret_cast<const int*>(w + L.rows);
    mp.chunk = chunk;
    mp.R = L.R;
    mp.S = S;
    mp.L = s.L;
    mp.V = s.V;
    mp.beta = s.beta;
    mp.loss_mode = s.loss_mode;
    mp.objective = s.objective;
    mp.seqcnt = reinterpret_cast<const int*>(w + L.seqcnt);
    mp.N = L.N;
    mp.lse = reinterpret_cast<float*>(w + L.lse);
    mp.gco = reinterpret_cast<float*>(w + L.gco);
    mp.ell = reinterpret_cast<float*>(w + L.ell);
    mp.row_stats = in.row_stats;
    mp.status = in.status;
    mp.rmax = nullptr;
    return mp;
}

FwdParams fwd_params(const Inputs& in, const WsLayout& L, char* w) {
    const grpo_shape& s = *in.shape;
    FwdParams fp = {};
    fp.counts = reinterpret_cast<const int*>(w + L.counts);
    fp.rows = reinterpret_cast<const int*>(w + L.rows);
    fp.tokens = in.tokens;
    fp.zt = reinterpret_cast<float2*>(w + L.zt);
    fp.N = L.N;
    fp.V = s.V;
    fp.d = s.d;
    fp.n_ntiles = L.n_ntiles;
    fp.V_pad = L.V_pad;
    fp.nc32 = L.nc32;
    fp.zscale[0] = fp.zscale[1] = 1.f;
    fp.status = in.status;
    return fp;
}

int run_index(const Inputs& in, const WsLayout& L, char* w, cudaStream_t st) {
    if (launch(GRPO_PROF_INDEX, st, [&] {
            return launch_index(in.mask, L.N, L.R, reinterpret_cast<int*>(w + L.counts),
                                reinterpret_cast<int*>(w + L.rows), reinterpret_cast<int2*>(w + L.tiles),
                                reinterpret_cast<int*>(w + L.sched), L.n_sched, in.status, st);
        }) != cudaSuccess)
        return GRPO_ERR_LAUNCH;
    if (in.shape->loss_mode == GRPO_SEQUENCE_MEAN &&
        launch(GRPO_PROF_INDEX, st, [&] {
            return launch_seq_counts(in.mask, L.n_seq, in.shape->L, reinterpret_cast<int*>(w + L.seqcnt),
                                     reinterpret_cast<int*>(w + L.counts), st);
        }) != cudaSuccess)
        return GRPO_ERR_LAUNCH;
    if (in.global_counts &&
        launch(GRPO_PROF_INDEX, st, [&] {
            return launch_apply_global_counts(in.global_counts, reinterpret_cast<int*>(w + L.counts),
                                              in.shape->loss_mode, in.status, st);
        }) != cudaSuccess)
        return GRPO_ERR_LAUNCH;
    return GRPO_OK;
}

int run_loss_reduce(const Inputs& in, const WsLayout& L, char* w, cudaStream_t st) {
    return launch(GRPO_PROF_MERGE, st, [&] {
               return launch_loss_reduce(reinterpret_cast<const float*>(w + L.ell), L.N,
                                         reinterpret_cast<double*>(w + L.blocksum), L.nblk,
                                         reinterpret_cast<const int*>(w + L.counts), in.loss_out, st);
           }) == cudaSuccess
               ? GRPO_OK
               : GRPO_ERR_LAUNCH;
}

// Forward over all rows at once: row tiles of h_pol / h_ref, per-row merge,
// loss reduction.  Touches only the workspace below the chunk buffers.
int run_forward(const Inputs& in, const WsLayout& L, const DeviceInfo& dev, cudaStream_t st) {
    const grpo_shape& s = *in.shape;
    const bool bf16 = s.dtype == GRPO_BF16;
    char* w = static_cast<char*>(in.ws);
    int rc = run_index(in, L, w, st);
    if (rc != GRPO_OK) return rc;
    CUtensorMap mHp, mHr, mW;
    if (!make_map(&mHp, in.h_pol, bf16, s.d, L.N, s.d, kBK, kBM) ||
        !make_map(&mHr, in.h_ref, bf16, s.d, L.N, s.d, kBK, kBM) ||
        !make_map(&mW, in.W, bf16, s.d, s.V, s.d, kBK, kBN))
        return GRPO_ERR_LAUNCH;
    FwdParams fp = fwd_params(in, L, w);
    fp.tiles = reinterpret_cast<const int2*>(w + L.tiles);
    fp.part = reinterpret_cast<float4*>(w + L.part);
    fp.S = L.S;
    fp.nps = L.nps;
    fp.sched = reinterpret_cast<int*>(w + L.sched);
    fp.chunk = -1;
    if (launch(GRPO_PROF_FWD, st, [&] { return launch_fwd(fp, mHp, mHr, mW, dev.sm_count, bf16, st); }) !=
        cudaSuccess)
        return GRPO_ERR_LAUNCH;
    const MergeParams mp = merge_params(in, L, w, -1, reinterpret_cast<const float4*>(w + L.part), L.S);
    if (launch(GRPO_PROF_MERGE, st, [&] { return launch_merge(mp, st); }) != cudaSuccess) return GRPO_ERR_LAUNCH;
    return run_loss_reduce(in, L, w, st);
}

// The chunked path: for each chunk of masked-in rows, gather compact copies of
// its h_pol / h_ref rows, run the SM-pair forward, merge per row; with a
// backward, keep the policy exponentials and turn them into dlogits, dH and
// dW.  Then reduce the loss.  Uses the whole workspace.
struct Backward {
    float loss_scale;
    void* dH;
    float* dW;
    int32_t* found_inf;
};

// 8-bit inputs: the format and the per-tensor scales
struct Fp8Inputs {
    bool e5m2;
    float h_pol, h_ref, w;
};

int run_chunked(const Inputs& in, const WsLayout& L, const DeviceInfo& dev, cudaStream_t st, const Backward* bwd,
                const Fp8Inputs* f8 = nullptr) {
    const grpo_shape& s = *in.shape;
    const bool bf16 = s.dtype == GRPO_BF16;
    const int row_bytes = f8 ? s.d : 2 * s.d;
    char* w = static_cast<char*>(in.ws);
    int* counts = reinterpret_cast<int*>(w + L.counts);
    int rc = run_index(in, L, w, st);
    if (rc != GRPO_OK) return rc;
    // masked rows: objective 0; with a backward: found_inf <- 0, dW <- 0 when no row
    // is masked in, dH rows of masked rows <- 0
    if (launch(GRPO_PROF_CLEAR, st, [&] {
            return launch_rows_init(in.mask, L.N, reinterpret_cast<float*>(w + L.ell), in.row_stats, dev.sm_count, st);
        }) != cudaSuccess)
        return GRPO_ERR_LAUNCH;
    if (bwd) {
        if (launch(GRPO_PROF_CLEAR, st, [&] {
                return launch_clear_grads(counts, bwd->found_inf, bwd->dW, static_cast<int64_t>(s.V) * s.d,
                                          dev.sm_count, st);
            }) != cudaSuccess)
            return GRPO_ERR_LAUNCH;
        if (launch(GRPO_PROF_CLEAR, st, [&] {
                return launch_zero_masked_rows(in.mask, L.N, s.d, bwd->dH, dev.sm_count, st);
            }) != cudaSuccess)
            return GRPO_ERR_LAUNCH;
    }

    CUtensorMap mW_k, mW_mn, mHc_k, mHcr_k, mHc_mn, mDS_k, mDS_mn;
    void* hc = w + L.hc;
    void* hcr = w + L.hcr;
    void* ds = w + L.ds;
    // W tiles for the pair forward: each CTA of a pair loads 128 of the 256 vocabulary rows
    if (f8) {
        // 8-bit inputs: a K-stage is one 128-byte span of 128 elements
        if (!make_map_u8(&mW_k, in.W, s.d, s.V, s.d, 128, kBN / 2) ||
            !make_map_u8(&mHc_k, hc, s.d, L.R, s.d, 128, kBM) || !make_map_u8(&mHcr_k, hcr, s.d, L.R, s.d, 128, kBM))
            return GRPO_ERR_LAUNCH;
        // the 8-bit backward: codes of the dlogits' softmax part K-major for dH, MN-major for dW;
        // W and the compact h_pol rows MN-major (128 x 128-byte boxes)
        if (bwd && (!make_map_u8(&mDS_k, w + L.qa, s.V, L.R, L.V_pad, 128, 128) ||
                    !make_map_u8(&mDS_mn, w + L.qb, s.V, L.R, L.V_pad, 128, 128) ||
                    !make_map_u8(&mW_mn, in.W, s.d, s.V, s.d, 128, 128) ||
                    !make_map_u8(&mHc_mn, hc, s.d, L.R, s.d, 128, 128)))
            return GRPO_ERR_LAUNCH;
    } else if (!make_map(&mW_k, in.W, bf16, s.d, s.V, s.d, kBK, kBN / 2) ||
               !make_map(&mW_mn, in.W, bf16, s.d, s.V, s.d, 64, kBK) ||
               !make_map(&mHc_k, hc, bf16, s.d, L.R, s.d, kBK, kBM) ||
               !make_map(&mHcr_k, hcr, bf16, s.d, L.R, s.d, kBK, kBM) ||
               !make_map(&mHc_mn, w + L.hct, bf16, L.R, s.d, L.R, kBK, 128) ||
               !make_map(&mDS_k, ds, bf16, s.V, L.R, L.V_pad, kBK, kBM) ||
               !make_map(&mDS_mn, ds, bf16, s.V, L.R, L.V_pad, 64, kBK)) {
        return GRPO_ERR_LAUNCH;
    }

    FwdParams fp = fwd_params(in, L, w);
    fp.tiles = nullptr;                                  // chunk mode
    fp.part = reinterpret_cast<float4*>(w + L.partc);
    fp.S = L.Sc;
    fp.nps = L.npsc;
    fp.R = L.R;
    // the exponentials are kept only when a backward follows
    fp.E = bwd ? static_cast<uint16_t*>(ds) : nullptr;
    fp.mx = bwd ? reinterpret_cast<float*>(w + L.mx) : nullptr;
    if (f8) {
        fp.zscale[0] = f8->h_pol * f8->w;
        fp.zscale[1] = f8->h_ref * f8->w;
    }

    ChunkParams cp;
    cp.counts = counts;
    cp.rows = reinterpret_cast<const int*>(w + L.rows);
    cp.tokens = in.tokens;
    cp.lse = reinterpret_cast<const float*>(w + L.lse);
    cp.gco = reinterpret_cast<const float*>(w + L.gco);
    cp.zt = reinterpret_cast<const float2*>(w + L.zt);
    cp.mx = reinterpret_cast<const float*>(w + L.mx);
    cp.scale = bwd ? bwd->loss_scale : 1.f;
    cp.V = s.V;
    cp.d = s.d;
    cp.V_pad = L.V_pad;
    cp.nc32 = L.nc32;
    cp.R = L.R;
    cp.N = L.N;
    cp.dS = static_cast<uint16_t*>(ds);
    cp.dH = bwd ? static_cast<uint16_t*>(bwd->dH) : nullptr;
    cp.dW = bwd ? bwd->dW : nullptr;
    cp.sched = nullptr;
    cp.found_inf = bwd ? bwd->found_inf : nullptr;
    cp.status = in.status;
    cp.qa = nullptr;
    cp.qb = nullptr;
    cp.rmax = nullptr;
    cp.gmax = nullptr;
    cp.keys = nullptr;
    cp.tokpos = nullptr;
    cp.hq = nullptr;
    cp.wq = nullptr;
    cp.scale_h = cp.scale_w = 1.f;
    cp.e5m2 = 0;
    if (f8 && bwd) {
        cp.qa = reinterpret_cast<uint8_t*>(w + L.qa);
        cp.qb = reinterpret_cast<uint8_t*>(w + L.qb);
        cp.rmax = reinterpret_cast<const float*>(w + L.rmax);
        cp.gmax = reinterpret_cast<float*>(w + L.gmax);
        cp.keys = reinterpret_cast<unsigned long long*>(w + L.keys);
        cp.tokpos = reinterpret_cast<int*>(w + L.tokpos);
        cp.hq = reinterpret_cast<const uint8_t*>(hc);
        cp.wq = static_cast<const uint8_t*>(in.W);
        cp.scale_h = f8->h_pol;
        cp.scale_w = f8->w;
        cp.e5m2 = f8->e5m2 ? 1 : 0;
    }
    const int64_t max_chunks = (L.N + L.R - 1) / L.R;
    // dH in 512-column units when a full chunk's units divide evenly over the SM pairs
    const int dh_pairs_of_tiles = (L.R / kBM + 1) / 2;
    const int dh_wide_tiles = (s.d + 2 * kBN - 1) / (2 * kBN);
    const bool dh_wide = (dh_pairs_of_tiles * dh_wide_tiles) % (dev.sm_count / 2) == 0;
    // 8-bit backward: every chunk's (token, slot) keys sorted at once, one block per chunk
    if (f8 && bwd && launch(GRPO_PROF_F8_PREP, st, [&] {
            return launch_sort_keys(cp, static_cast<int>(max_chunks), st);
        }) != cudaSuccess)
        return GRPO_ERR_LAUNCH;
    unsigned long long* keys_all = cp.keys;
    for (int64_t c = 0; c < max_chunks; ++c) {
        const int ci = static_cast<int>(c);
        cp.chunk = ci;
        if (keys_all) cp.keys = keys_all + c * L.R;
        fp.chunk = ci;
        fp.sched = reinterpret_cast<int*>(w + L.sched) + 1 + ci;
        MergeParams mp = merge_params(in, L, w, ci, reinterpret_cast<const float4*>(w + L.partc), L.Sc);
        if (f8 && bwd) mp.rmax = reinterpret_cast<float*>(w + L.rmax);
        if (launch(GRPO_PROF_GATHER, st, [&] {
                // 16-bit inputs with a backward also get the transposed compact h_pol rows (dW's B operand)
                return bwd && !f8 ? launch_gather_rows_t(cp, in.h_pol, hc, in.h_ref, hcr, w + L.hct, L.R,
                                                         dev.sm_count, st)
                                  : launch_gather_rows(cp, in.h_pol, hc, in.h_ref, hcr, L.R, row_bytes, dev.sm_count,
                                                       st);
            }) != cudaSuccess)
            return GRPO_ERR_LAUNCH;
        if (launch(GRPO_PROF_FWD, st, [&] {
                return f8 ? launch_fwd_pair_fp8(fp, mHc_k, mHcr_k, mW_k, dev.sm_count, f8->e5m2, st)
                          : launch_fwd_pair(fp, mHc_k, mHcr_k, mW_k, dev.sm_count, bf16, st);
            }) != cudaSuccess)
            return GRPO_ERR_LAUNCH;
        if (launch(GRPO_PROF_MERGE, st, [&] { return launch_merge(mp, st); }) != cudaSuccess) return GRPO_ERR_LAUNCH;
        if (!bwd) continue;
        if (f8) {
            if (launch(GRPO_PROF_F8_PREP, st, [&] { return launch_f8_group_max(cp, dev.sm_count, st); }) !=
                    cudaSuccess ||
                launch(GRPO_PROF_DLOGITS, st, [&] { return launch_transform_f8(cp, dev.sm_count, st); }) !=
                    cudaSuccess ||
                launch(GRPO_PROF_DH, st, [&] { return launch_dh_pair_fp8(cp, mDS_k, mW_mn, dev.sm_count, dh_wide, st); }) !=
                    cudaSuccess ||
                launch(GRPO_PROF_DW, st, [&] { return launch_dw_pair_fp8(cp, mDS_mn, mHc_mn, dev.sm_count, st); }) !=
                    cudaSuccess)
                return GRPO_ERR_LAUNCH;
            continue;
        }
        if (launch(GRPO_PROF_DLOGITS, st, [&] { return launch_transform(cp, bf16, L.R, dev.sm_count, st); }) !=
            cudaSuccess)
            return GRPO_ERR_LAUNCH;
        if (launch(GRPO_PROF_DH, st, [&] {
                return launch_dh_pair(cp, mDS_k, mW_mn, dev.sm_count, bf16, dh_wide, st);
            }) != cudaSuccess)
            return GRPO_ERR_LAUNCH;
        if (launch(GRPO_PROF_DW, st, [&] { return launch_dw_pair(cp, mDS_mn, mHc_mn, dev.sm_count, bf16, st); }) !=
            cudaSuccess)
            return GRPO_ERR_LAUNCH;
    }
    return run_loss_reduce(in, L, w, st);
}

}  // namespace

extern "C" {

void grpo_shape_init(grpo_shape* s, int n_groups, int G, int L, int d, int V, grpo_dtype dtype) {
    if (!s) return;
    std::memset(s, 0, sizeof(*s));
    s->n_groups = n_groups;
    s->G = G;
    s->L = L;
    s->d = d;
    s->V = V;
    s->dtype = dtype;
    s->beta = 0.04f;
    s->eps = 1e-4f;
    s->std_unbiased = 1;
    s->chunk_rows = 0;
    s->loss_mode = GRPO_TOKEN_MEAN;
    s->objective = GRPO_OBJ_GRPO;
}

int grpo_chunk_rows(const grpo_shape* shape) {
    if (!shape || !shape_ok(*shape)) return 0;
    return chunk_rows_of(*shape);
}

size_t grpo_workspace_bytes(const grpo_shape* shape) {
    if (!shape || !dtype_ok_any(*shape)) return 0;
    WsLayout L;
    if (!ws_layout(*shape, &L)) return 0;
    return L.total;
}

int grpo_group_advantages(const float* rewards, int n_groups, int G, float eps, int std_unbiased, float* adv_out,
                          grpo_stream_t stream) {
    if (n_groups < 1 || G < 1) return GRPO_ERR_SHAPE;
    if (!rewards || !adv_out || !aligned(rewards, 4) || !aligned(adv_out, 4)) return GRPO_ERR_POINTER;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return launch(GRPO_PROF_ADVANTAGES, st,
                  [&] { return launch_advantages(rewards, n_groups, G, eps, std_unbiased, adv_out, st); }) ==
                   cudaSuccess
               ? GRPO_OK
               : GRPO_ERR_LAUNCH;
}

int grpo_build_mask(const int32_t* lengths, const grpo_shape* shape, uint8_t* mask_out, grpo_stream_t stream) {
    if (!shape || !shape_ok(*shape)) return GRPO_ERR_SHAPE;
    if (!lengths || !mask_out || !aligned(lengths, 4)) return GRPO_ERR_POINTER;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return launch(GRPO_PROF_MASK, st,
                  [&] { return launch_build_mask(lengths, shape->n_groups * shape->G, shape->L, mask_out, st); }) ==
                   cudaSuccess
               ? GRPO_OK
               : GRPO_ERR_LAUNCH;
}

int grpo_valid_rows(const uint8_t* mask, const grpo_shape* shape, int32_t* rows_out, int32_t* n_valid_out,
                    void* workspace, size_t ws_bytes, grpo_stream_t stream) {
    if (!shape) return GRPO_ERR_SHAPE;
    WsLayout L;
    if (!ws_layout(*shape, &L)) return GRPO_ERR_SHAPE;
    if (!mask || !rows_out || !n_valid_out || !workspace) return GRPO_ERR_POINTER;
    if (!aligned(rows_out, 4) || !aligned(n_valid_out, 4) || !aligned(workspace, 256)) return GRPO_ERR_POINTER;
    if (ws_bytes < L.total) return GRPO_ERR_WORKSPACE;
    char* w = static_cast<char*>(workspace);
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    int* counts = reinterpret_cast<int*>(w + L.counts);
    int* scratch_status = counts + 8;
    if (launch(GRPO_PROF_INDEX, st, [&] {
            return launch_index(mask, L.N, L.R, counts, rows_out, reinterpret_cast<int2*>(w + L.tiles),
                                reinterpret_cast<int*>(w + L.sched), L.n_sched, scratch_status, st);
        }) != cudaSuccess)
        return GRPO_ERR_LAUNCH;
    if (cudaMemcpyAsync(n_valid_out, counts + C_NVALID, sizeof(int32_t), cudaMemcpyDeviceToDevice, st) != cudaSuccess)
        return GRPO_ERR_LAUNCH;
    return GRPO_OK;
}

int grpo_loss_fwd(const void* h_pol, const void* h_ref, const void* W, const int32_t* tokens, const uint8_t* mask,
                  const float* adv, const grpo_shape* shape, void* workspace, size_t ws_bytes, float* loss_out,
                  float* row_stats, int32_t* status, grpo_stream_t stream) {
    Inputs in{h_pol, h_ref, W, tokens, mask, adv, shape, workspace, ws_bytes, loss_out, row_stats, status};
    WsLayout L;
    int rc = validate(in, &L);
    if (rc != GRPO_OK) return rc;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != GRPO_OK) return rc;
    return run_chunked(in, L, dev, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

int grpo_loss_fwd_bwd(const void* h_pol, const void* h_ref, const void* W, const int32_t* tokens, const uint8_t* mask,
                      const float* adv, const grpo_shape* shape, float loss_scale, void* workspace, size_t ws_bytes,
                      float* loss_out, void* dH, float* dW, int32_t* found_inf, float* row_stats, int32_t* status,
                      grpo_stream_t stream) {
    Inputs in{h_pol, h_ref, W, tokens, mask, adv, shape, workspace, ws_bytes, loss_out, row_stats, status};
    WsLayout L;
    int rc = validate(in, &L);
    if (rc != GRPO_OK) return rc;
    if (!dH || !dW || !found_inf || !aligned(dH, 32) || !aligned(dW, 32) || !aligned(found_inf, 4))
        return GRPO_ERR_POINTER;
    if (!(loss_scale > 0.f) || !std::isfinite(loss_scale)) return GRPO_ERR_SHAPE;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != GRPO_OK) return rc;
    const Backward bwd{loss_scale, dH, dW, found_inf};
    return run_chunked(in, L, dev, reinterpret_cast<cudaStream_t>(stream), &bwd);
}

int grpo_shard_counts(const uint8_t* mask, const grpo_shape* shape, int32_t* counts_out, grpo_stream_t stream) {
    if (!shape || !shape_ok(*shape)) return GRPO_ERR_SHAPE;
    if (!mask || !counts_out || !aligned(counts_out, 4)) return GRPO_ERR_POINTER;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return launch(GRPO_PROF_INDEX, st, [&] {
               return launch_shard_counts(mask, shape->n_groups * shape->G, shape->L, counts_out, st);
           }) == cudaSuccess
               ? GRPO_OK
               : GRPO_ERR_LAUNCH;
}

int grpo_loss_fwd_shard(const void* h_pol, const void* h_ref, const void* W, const int32_t* tokens,
                        const uint8_t* mask, const float* adv, const grpo_shape* shape,
                        const int32_t* global_counts, void* workspace, size_t ws_bytes, float* loss_out,
                        float* row_stats, int32_t* status, grpo_stream_t stream) {
    Inputs in{h_pol, h_ref, W, tokens, mask, adv, shape, workspace, ws_bytes, loss_out, row_stats, status};
    in.global_counts = global_counts;
    WsLayout L;
    int rc = validate(in, &L);
    if (rc != GRPO_OK) return rc;
    if (!global_counts || !aligned(global_counts, 4)) return GRPO_ERR_POINTER;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != GRPO_OK) return rc;
    return run_chunked(in, L, dev, reinterpret_cast<cudaStream_t>(stream), nullptr);
}

int grpo_loss_fwd_bwd_shard(const void* h_pol, const void* h_ref, const void* W, const int32_t* tokens,
                            const uint8_t* mask, const float* adv, const grpo_shape* shape,
                            const int32_t* global_counts, float loss_scale, void* workspace, size_t ws_bytes,
                            float* loss_out, void* dH, float* dW, int32_t* found_inf, float* row_stats,
                            int32_t* status, grpo_stream_t stream) {
    Inputs in{h_pol, h_ref, W, tokens, mask, adv, shape, workspace, ws_bytes, loss_out, row_stats, status};
    in.global_counts = global_counts;
    WsLayout L;
    int rc = validate(in, &L);
    if (rc != GRPO_OK) return rc;
    if (!global_counts || !aligned(global_counts, 4)) return GRPO_ERR_POINTER;
    if (!dH || !dW || !found_inf || !aligned(dH, 32) || !aligned(dW, 32) || !aligned(found_inf, 4))
        return GRPO_ERR_POINTER;
    if (!(loss_scale > 0.f) || !std::isfinite(loss_scale)) return GRPO_ERR_SHAPE;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != GRPO_OK) return rc;
    const Backward bwd{loss_scale, dH, dW, found_inf};
    return run_chunked(in, L, dev, reinterpret_cast<cudaStream_t>(stream), &bwd);
}

// Shared argument checks of the two 8-bit entry points; on success *L is the
// 8-bit workspace layout and *s16 the shape the 16-bit steps run with.
static int validate_fp8(const Inputs& in8, float scale_h_pol, float scale_h_ref, float scale_w, WsLayout* L,
                        grpo_shape* s16) {
    if (!in8.shape) return GRPO_ERR_SHAPE;
    const grpo_shape& s = *in8.shape;
    if (!is_fp8(s.dtype)) return GRPO_ERR_DTYPE;
    if (s.d % 128 != 0) return GRPO_ERR_SHAPE;
    if (!(scale_h_pol > 0.f) || !(scale_h_ref > 0.f) || !(scale_w > 0.f) || !std::isfinite(scale_h_pol) ||
        !std::isfinite(scale_h_ref) || !std::isfinite(scale_w))
        return GRPO_ERR_SHAPE;
    if (!ws_layout(s, L)) return GRPO_ERR_SHAPE;
    *s16 = s;
    s16->dtype = GRPO_BF16;
    // the pointer and shape checks of the 16-bit path; the workspace is checked against the 8-bit layout
    Inputs in = in8;
    in.shape = s16;
    in.ws_bytes = ~static_cast<size_t>(0);
    WsLayout L16;
    const int rc = validate(in, &L16);
    if (rc != GRPO_OK) return rc;
    if (in8.ws_bytes < L->total) return GRPO_ERR_WORKSPACE;
    return GRPO_OK;
}

int grpo_loss_fwd_fp8(const void* h_pol, const void* h_ref, const void* W, float scale_h_pol, float scale_h_ref,
                      float scale_w, const int32_t* tokens, const uint8_t* mask, const float* adv,
                      const grpo_shape* shape, void* workspace, size_t ws_bytes, float* loss_out, float* row_stats,
                      int32_t* status, grpo_stream_t stream) {
    Inputs in{h_pol, h_ref, W, tokens, mask, adv, shape, workspace, ws_bytes, loss_out, row_stats, status};
    WsLayout L;
    grpo_shape s16;
    int rc = validate_fp8(in, scale_h_pol, scale_h_ref, scale_w, &L, &s16);
    if (rc != GRPO_OK) return rc;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != GRPO_OK) return rc;
    in.shape = &s16;
    const Fp8Inputs f8{shape->dtype == GRPO_E5M2, scale_h_pol, scale_h_ref, scale_w};
    return run_chunked(in, L, dev, reinterpret_cast<cudaStream_t>(stream), nullptr, &f8);
}

int grpo_loss_fwd_bwd_fp8(const void* h_pol, const void* h_ref, const void* W, float scale_h_pol, float scale_h_ref,
                          float scale_w, const int32_t* tokens, const uint8_t* mask, const float* adv,
                          const grpo_shape* shape, void* workspace, size_t ws_bytes, float* loss_out, void* dH,
                          float* dW, float* row_stats, int32_t* status, grpo_stream_t stream) {
    Inputs in{h_pol, h_ref, W, tokens, mask, adv, shape, workspace, ws_bytes, loss_out, row_stats, status};
    WsLayout L;
    grpo_shape s16;
    int rc = validate_fp8(in, scale_h_pol, scale_h_ref, scale_w, &L, &s16);
    if (rc != GRPO_OK) return rc;
    if (L.R > kF8SortMax) return GRPO_ERR_SHAPE;
    if (!dH || !dW || !aligned(dH, 32) || !aligned(dW, 32)) return GRPO_ERR_POINTER;
    DeviceInfo dev;
    rc = device_info(&dev);
    if (rc != GRPO_OK) return rc;
    in.shape = &s16;
    // no loss scaling on this path (dH is bf16): found_inf goes to a spare workspace word
    int32_t* spare_inf = reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + L.counts) + C_SPARE_INF;
    const Backward bwd{1.f, dH, dW, spare_inf};
    const Fp8Inputs f8{shape->dtype == GRPO_E5M2, scale_h_pol, scale_h_ref, scale_w};
    return run_chunked(in, L, dev, reinterpret_cast<cudaStream_t>(stream), &bwd, &f8);
}

int grpo_device_checks(void) {
#ifdef GRPO_DEVICE_CHECKS
    return 1;
#else
    return 0;
#endif
}

int grpo_selftest_bounds_check(int32_t* status, grpo_stream_t stream) {
    if (!status || !aligned(status, 4)) return GRPO_ERR_POINTER;
#ifdef GRPO_DEVICE_CHECKS
    DeviceInfo dev;
    const int rc = device_info(&dev);
    if (rc != GRPO_OK) return rc;
    if (launch_bounds_selftest(status, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return GRPO_ERR_LAUNCH;
    return GRPO_OK;
#else
    (void)stream;
    return GRPO_ERR_DEVICE;   // built without device checks: nothing is launched
#endif
}

int grpo_selftest_wait_timeout(int32_t* status, unsigned long long* waited_ns, grpo_stream_t stream) {
    if (!status || !waited_ns || !aligned(status, 4) || !aligned(waited_ns, 8)) return GRPO_ERR_POINTER;
    DeviceInfo dev;
    const int rc = device_info(&dev);
    if (rc != GRPO_OK) return rc;
    return launch_wait_selftest(status, waited_ns, reinterpret_cast<cudaStream_t>(stream)) == cudaSuccess
               ? GRPO_OK
               : GRPO_ERR_LAUNCH;
}

const char* grpo_status_string(int status) {
    switch (status) {
        case GRPO_OK: return "ok";
        case GRPO_ERR_POINTER: return "null or misaligned pointer";
        case GRPO_ERR_SHAPE: return "bad shape or token id";
        case GRPO_ERR_WORKSPACE: return "workspace too small";
        case GRPO_ERR_LAUNCH: return "CUDA launch or driver error";
        case GRPO_ERR_DTYPE: return "unsupported dtype";
        case GRPO_ERR_TIMEOUT: return "device wait timed out";
        case GRPO_ERR_DEVICE: return "device is not an sm_103 GPU with enough shared memory";
        case GRPO_ERR_BOUNDS: return "device index check failed (checked build)";
        default: return "unknown status";
    }
}

int grpo_version(void) { return kVersion; }

int grpo_profile_enable(int on) {
    g_prof.on.store(on != 0);
    return GRPO_OK;
}

int grpo_profile_collect(double* ms, long long* launches, int n_kinds) {
    if ((!ms || !launches) && n_kinds > 0) return GRPO_ERR_POINTER;
    std::lock_guard<std::mutex> lock(g_prof.mu);
    int rc = GRPO_OK;
    for (const ProfRecord& r : g_prof.recs) {
        float t = 0.f;
        if (cudaEventSynchronize(r.b) != cudaSuccess || cudaEventElapsedTime(&t, r.a, r.b) != cudaSuccess)
            rc = GRPO_ERR_LAUNCH;
        if (r.kind < n_kinds) {
            ms[r.kind] += static_cast<double>(t);
            launches[r.kind] += 1;
        }
        g_prof.pool.push_back(r.a);
        g_prof.pool.push_back(r.b);
    }
    g_prof.recs.clear();
    return rc;
}

unsigned long long grpo_kernel_launches(void) { return g_launches.load(); }

}  // extern "C"

// ---------------------------------------------------------------------------
// Forward loss without a caller-provided workspace.
//
// Some callers cannot allocate device memory when they need the loss: a
// training step that runs next to an inference engine which has reserved all
// free device memory for its own pool ("Long-context GRPO", section 2 (3):
// training and vLLM inference share one memory space), or code that must not pay for cudaMalloc's
// device-wide synchronisation inside its step.  This entry point serves them
// from a fixed array that lives in the library itself.
namespace {

constexpr size_t kNoAllocScratchBytes = static_cast<size_t>(8) << 20;   // 8 MiB on every device
constexpr int64_t kNoAllocMaxRows = 32768;                                // n_groups * G * L
constexpr int kNoAllocMaxDevices = 256;

// The forward's workspace.  Every GPU that loads the library holds these
// 8 MiB until the process exits.  In host code the name is only a handle:
// kernels get the device address looked up below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_noalloc_mu;
void* g_noalloc_addr[kNoAllocMaxDevices] = {};

// Device address of the array on the current device, looked up once per device.
int noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return GRPO_ERR_LAUNCH;
    if (dev < 0 || dev >= kNoAllocMaxDevices) return GRPO_ERR_DEVICE;
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_addr[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p) return GRPO_ERR_LAUNCH;
        g_noalloc_addr[dev] = p;
    }
    *out = g_noalloc_addr[dev];
    return GRPO_OK;
}

}  // namespace

extern "C" int grpo_loss_fwd_noalloc(const void* h_pol, const void* h_ref, const void* W, const int32_t* tokens,
                                     const uint8_t* mask, const float* adv, const grpo_shape* shape,
                                     float* loss_out, float* row_stats, int32_t* status, grpo_stream_t stream) {
    if (!shape) return GRPO_ERR_SHAPE;
    if (!dtype_ok(*shape)) return GRPO_ERR_DTYPE;
    WsLayout L;
    if (!ws_layout(*shape, &L)) return GRPO_ERR_SHAPE;
    // the forward only touches the workspace below the backward buffers (L.hc)
    if (L.N > kNoAllocMaxRows || L.hc > kNoAllocScratchBytes) return GRPO_ERR_WORKSPACE;
    if (!h_pol || !h_ref || !W || !tokens || !mask || !adv || !loss_out || !status) return GRPO_ERR_POINTER;
    if (!aligned(h_pol, 16) || !aligned(h_ref, 16) || !aligned(W, 16) || !aligned(tokens, 4) || !aligned(adv, 4) ||
        !aligned(loss_out, 4) || !aligned(status, 4) || (row_stats && !aligned(row_stats, 4)))
        return GRPO_ERR_POINTER;
    DeviceInfo dev;
    int rc = device_info(&dev);
    if (rc != GRPO_OK) return rc;
    void* scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc != GRPO_OK) return rc;
    // Nothing in the array needs clearing: every word the forward reads is
    // written earlier in the same call (row index, per-split partials of the
    // masked-in rows, per-block sums).
    Inputs in{h_pol, h_ref, W, tokens, mask, adv, shape, scratch, L.hc, loss_out, row_stats, status};
    return run_forward(in, L, dev, reinterpret_cast<cudaStream_t>(stream));
}
