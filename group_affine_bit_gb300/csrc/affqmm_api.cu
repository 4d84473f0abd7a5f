// affqmm_api.cu -- the C ABI of libaffqmm: host-side validation, the work
// decomposition and the launches.  See include/affqmm.h for the contract.
#include <cuda.h>
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>

#include "affqmm.h"
#include "affqmm_format.cuh"
#include "affqmm_internal.h"

using namespace affqmm;

namespace {

constexpr int kMaxDevices = 64;

bool valid_bits(int b) { return b == 2 || b == 3 || b == 4 || b == 5 || b == 6 || b == 8; }
bool valid_group(int g) { return g == 32 || g == 64 || g == 128; }
bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Per-device facts the decomposition depends on (a cache of queries, not state
// that changes what a call computes on a given device).
struct DeviceInfo {
    int dev = 0;
    int sms = 0;
    int dec_ctas_per_sm = 0;  // decode CTAs resident per SM
    bool ok = false;
    bool is_sm103 = false;
};
DeviceInfo g_dev[kMaxDevices];
std::once_flag g_once[kMaxDevices];

int device_info(DeviceInfo** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return AFFQMM_E_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return AFFQMM_E_DEVICE;
    std::call_once(g_once[dev], [dev] {
        DeviceInfo& d = g_dev[dev];
        d.dev = dev;
        cudaDeviceProp prop;
        if (cudaGetDeviceProperties(&prop, dev) != cudaSuccess) return;
        d.sms = prop.multiProcessorCount;
        d.is_sm103 = prop.major == 10 && prop.minor == 3;
        if (!d.is_sm103) { d.ok = true; return; }
        if (decode_allow_smem(&d.dec_ctas_per_sm) != cudaSuccess) return;
        if (prompt_allow_smem() != cudaSuccess) return;
        d.ok = true;
    });
    DeviceInfo& d = g_dev[dev];
    if (!d.ok) return AFFQMM_E_CUDA;
    if (!d.is_sm103) return AFFQMM_E_DEVICE;
    *out = &d;
    return AFFQMM_OK;
}

int check_weight(const affqmm_weight* w) {
    if (!w) return AFFQMM_E_NULL;
    if (!valid_bits(w->bits)) return AFFQMM_E_BITS;
    if (!valid_group(w->group)) return AFFQMM_E_GROUP;
    if (w->N < 0 || w->K < 0 || (w->K % w->group) != 0) return AFFQMM_E_SHAPE;
    if (w->N > (int64_t)1 << 34 || w->K > (int64_t)1 << 28) return AFFQMM_E_SHAPE;
    const int64_t tiles = (w->N + TILE_N - 1) / TILE_N;
    const int64_t kb = (w->K + KBLK - 1) / KBLK;
    if (tiles * kb > ((int64_t)1 << 31) - 1) return AFFQMM_E_SHAPE;
    if (w->N > 0 && w->K > 0) {
        if (!w->packed) return AFFQMM_E_NULL;
        if (!aligned(w->packed, 256)) return AFFQMM_E_ALIGN;
    }
    return AFFQMM_OK;
}

void bind_workspace(DecodePlan* plan, void* workspace) {
    if (plan->ws_bytes == 0) return;
    uint8_t* base = static_cast<uint8_t*>(workspace);
    plan->p.status = reinterpret_cast<uint32_t*>(base);
    plan->p.counters = reinterpret_cast<uint32_t*>(base + kStatusBytes);
    plan->p.partials = reinterpret_cast<float*>(base + kSlotsOffset);
}


// cuTensorMapEncodeTiled, fetched from the driver at run time.
using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_tiled() {
    static EncodeTiledFn fn = [] {
        void* f = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
                cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return (EncodeTiledFn) nullptr;
        return reinterpret_cast<EncodeTiledFn>(f);
    }();
    return fn;
}

// The driver's asynchronous host<->device copies, fetched at run time like
// the tensor-map encoder: the driver, which registered the caller's
// page-locked buffers, decides whether a copy can run asynchronously.
using CopyHtoDFn = CUresult (*)(CUdeviceptr, const void*, size_t, CUstream);
using CopyDtoHFn = CUresult (*)(void*, CUdeviceptr, size_t, CUstream);
template <typename Fn>
Fn driver_fn(const char* name) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion(name, &f, 12000, cudaEnableDefault, &q) != cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
        return nullptr;
    return reinterpret_cast<Fn>(f);
}
// The GPU's address of page-locked host memory, or NULL for any other memory
// (pageable host memory, device memory, an unknown pointer).
using PointerAttrFn = CUresult (*)(void*, CUpointer_attribute, CUdeviceptr);
const void* host_on_device(const void* p) {
    static PointerAttrFn get = driver_fn<PointerAttrFn>("cuPointerGetAttribute");
    if (!get || !p) return nullptr;
    unsigned int type = 0;
    if (get(&type, CU_POINTER_ATTRIBUTE_MEMORY_TYPE, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS ||
        type != CU_MEMORYTYPE_HOST)
        return nullptr;
    CUdeviceptr d = 0;
    if (get(&d, CU_POINTER_ATTRIBUTE_DEVICE_POINTER, reinterpret_cast<CUdeviceptr>(p)) != CUDA_SUCCESS) return nullptr;
    return reinterpret_cast<const void*>(d);
}

CopyHtoDFn copy_htod() {
    static CopyHtoDFn fn = driver_fn<CopyHtoDFn>("cuMemcpyHtoDAsync");
    return fn;
}
CopyDtoHFn copy_dtoh() {
    static CopyDtoHFn fn = driver_fn<CopyDtoHFn>("cuMemcpyDtoHAsync");
    return fn;
}

// x [M, K] bf16 row-major as 64 (k) x 128-row boxes with the 128-byte
// swizzle the tensor core reads (the prompt kernel); rows past M and k past
// K read as zero.
int make_x_map(const uint16_t* x, int64_t M, int64_t K, int box_rows, CUtensorMap* map) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return AFFQMM_E_CUDA;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {64, (cuuint32_t)box_rows};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? AFFQMM_OK : AFFQMM_E_CUDA;
}

// x [M, K] bf16 for the decode kernel: boxes of 136 k x M rows, unswizzled,
// so a block's tile lands as M rows of 272 bytes (its 128 k and 8 of the next
// block, which the kernel does not use); k past K reads as zero.
int make_x_map_decode(const uint16_t* x, int64_t M, int64_t K, CUtensorMap* map) {
    EncodeTiledFn fn = encode_tiled();
    if (!fn) return AFFQMM_E_CUDA;
    const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)M};
    const cuuint64_t strides[1] = {(cuuint64_t)K * 2};
    const cuuint32_t box[2] = {136, (cuuint32_t)M};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<uint16_t*>(x), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? AFFQMM_OK : AFFQMM_E_CUDA;
}

int workspace_for(int count, const affqmm_weight* ws, int64_t M, size_t* bytes) {
    DeviceInfo* d = nullptr;
    int rc = device_info(&d);
    if (rc) return rc;
    *bytes = 0;
    if (M == 0) return AFFQMM_OK;
    if (M <= kDecodeRows) {
        DecodePlan plan;
        rc = plan_decode(d->sms, d->dec_ctas_per_sm, count, ws, M, &plan);
        if (rc) return rc;
        *bytes = plan.ws_bytes;
    } else {
        PromptPlan plan;
        rc = plan_prompt(d->sms, count, ws, std::min<int64_t>(M, kPromptRows), &plan);
        if (rc) return rc;
        *bytes = plan.ws_bytes;
    }
    return AFFQMM_OK;
}

int check_stack(int count, const affqmm_weight* ws) {
    if (count < 1 || count > AFFQMM_MAX_STACK) return AFFQMM_E_ARG;
    if (!ws) return AFFQMM_E_NULL;
    for (int i = 0; i < count; ++i) {
        int rc = check_weight(&ws[i]);
        if (rc) return rc;
        if (ws[i].K != ws[0].K || ws[i].bits != ws[0].bits || ws[i].group != ws[0].group) return AFFQMM_E_ARG;
    }
    return AFFQMM_OK;
}

int check_workspace(size_t need, void* workspace, size_t ws_bytes) {
    if (need == 0) return AFFQMM_OK;
    if (!workspace || ws_bytes < need) return AFFQMM_E_WORKSPACE;
    if (!aligned(workspace, 256)) return AFFQMM_E_ALIGN;
    return AFFQMM_OK;
}

// Validate everything, plan, and (unless `dry`) enqueue the launches.  A dry
// run returns the status the real call would return before any launch.
// Options of the decode-only forms: exact codes, the caller's group sums of
// x, the GeGLU epilogue.
struct Form {
    bool exact = false;
    const float* xsums = nullptr;
    int epi = 0;
};

// A per-thread cache of finished single-launch set-ups (the plan, bound to
// its workspace and outputs, and the encoded x tensor map): a call whose
// arguments equal an earlier call's -- the usual case in a decode loop, and
// the dry run that affqmm_run_host makes before its real call -- skips the
// planning and the encoding.  The set-up depends only on the arguments'
// values (shapes, pointers, the device), never on the memory they point to.
struct LaunchKey {
    int dev;
    int count;
    int epi;
    int exact;
    int64_t M;
    const void* x;
    const void* xsums;
    const void* workspace;
    size_t ws_bytes;
    affqmm_weight w[AFFQMM_MAX_STACK];
    uint16_t* ys[AFFQMM_MAX_STACK];
};
struct CachedLaunch {
    bool valid = false;
    bool decode = false;
    LaunchKey key;
    DecodePlan dplan;
    PromptPlan pplan;
    CUtensorMap map;
};
constexpr int kLaunchCache = 4;
thread_local CachedLaunch t_cache[kLaunchCache];
thread_local int t_cache_next = 0;

void make_key(LaunchKey* k, int dev, int count, const affqmm_weight* ws, const uint16_t* x, int64_t M,
              uint16_t* const* ys, void* workspace, size_t ws_bytes, const Form& form) {
    std::memset(k, 0, sizeof(*k));  // padding included: keys are compared bytewise
    k->dev = dev;
    k->count = count;
    k->epi = form.epi;
    k->exact = form.exact ? 1 : 0;
    k->M = M;
    k->x = x;
    k->xsums = form.xsums;
    k->workspace = workspace;
    k->ws_bytes = ws_bytes;
    for (int i = 0; i < count; ++i) {
        k->w[i] = ws[i];
        k->ys[i] = ys[i];
    }
}

CachedLaunch* find_launch(const LaunchKey& k) {
    for (CachedLaunch& c : t_cache)
        if (c.valid && std::memcmp(&c.key, &k, sizeof k) == 0) return &c;
    return nullptr;
}

CachedLaunch* new_launch(const LaunchKey& k) {
    CachedLaunch& c = t_cache[t_cache_next];
    t_cache_next = (t_cache_next + 1) % kLaunchCache;
    c.valid = false;
    c.key = k;
    return &c;
}

int run_impl(int count, const affqmm_weight* ws, const uint16_t* x, int64_t M, uint16_t* const* ys,
             void* workspace, size_t ws_bytes, void* stream, Form form = Form(), bool dry = false) {
    int rc = check_stack(count, ws);
    if (rc) return rc;
    const bool decode_only = form.exact || form.epi != 0;
    if (M < 0 || M > AFFQMM_MAX_M || (decode_only && M > kDecodeRows)) return AFFQMM_E_M;
    if (form.epi != 0)
        for (int i = 0; i < count; ++i)
            if (ws[i].N % 32 != 0) return AFFQMM_E_SHAPE;  // gate/up rows interleaved in 16-row blocks
    if (form.xsums && !aligned(form.xsums, 4)) return AFFQMM_E_ALIGN;
    if (M == 0) return AFFQMM_OK;
    const int64_t K = ws[0].K;
    int64_t total_n = 0;
    for (int i = 0; i < count; ++i) {
        total_n += ws[i].N;
        if (ws[i].N > 0 && !ys[i]) return AFFQMM_E_NULL;
        if (ys[i] && !aligned(ys[i], 2)) return AFFQMM_E_ALIGN;
    }
    if (total_n == 0) return AFFQMM_OK;
    if (K > 0) {
        if (!x) return AFFQMM_E_NULL;
        if (!aligned(x, 16)) return AFFQMM_E_ALIGN;
    }
    DeviceInfo* d = nullptr;
    rc = device_info(&d);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (K == 0) {  // an empty sum: every output is +0
        if (dry) return AFFQMM_OK;
        for (int i = 0; i < count; ++i)
            if (ws[i].N > 0 && cudaMemsetAsync(ys[i], 0, (size_t)M * ws[i].N * 2 / (form.epi ? 2 : 1), st) != cudaSuccess)
                return AFFQMM_E_CUDA;
        return AFFQMM_OK;
    }
    LaunchKey key;
    make_key(&key, d->dev, count, ws, x, M, ys, workspace, ws_bytes, form);
    if (M <= kDecodeRows) {
        CachedLaunch* c = find_launch(key);
        if (!c) {
            DecodePlan plan;
            rc = plan_decode(d->sms, d->dec_ctas_per_sm, count, ws, M, &plan);
            if (rc) return rc;
            rc = check_workspace(plan.ws_bytes, workspace, ws_bytes);
            if (rc) return rc;
            bind_workspace(&plan, workspace);
            for (int i = 0; i < count; ++i) plan.p.proj[i].y = ys[i];
            plan.p.x = x;
            plan.p.xsums = form.xsums;
            plan.p.epi = form.epi;
            CUtensorMap map;
            rc = make_x_map_decode(x, M, K, &map);
            if (rc) return rc;
            c = new_launch(key);
            c->decode = true;
            c->dplan = plan;
            c->map = map;
            c->valid = true;
        }
        if (dry) return AFFQMM_OK;
        c->dplan.p.fault_wait = decode_fault_wait();  // the test hook's current setting
        if (launch_decode(ws[0].bits, ws[0].group, c->dplan.p, c->map, c->dplan.grid, st, form.exact) !=
            cudaSuccess)
            return AFFQMM_E_CUDA;
        return AFFQMM_OK;
    }
    if (M <= kPromptRows) {  // one prompt launch
        CachedLaunch* c = find_launch(key);
        if (!c) {
            PromptPlan plan;
            rc = plan_prompt(d->sms, count, ws, M, &plan);
            if (rc) return rc;
            rc = check_workspace(plan.ws_bytes, workspace, ws_bytes);
            if (rc) return rc;
            uint8_t* wsb = static_cast<uint8_t*>(workspace);
            plan.p.status = reinterpret_cast<uint32_t*>(wsb);
            plan.p.counters = reinterpret_cast<uint32_t*>(wsb + kStatusBytes);
            plan.p.slots = reinterpret_cast<float*>(wsb + kSlotsOffset);
            for (int i = 0; i < count; ++i) plan.p.proj[i].y = ys[i];
            CUtensorMap map;
            rc = make_x_map(x, M, K, 128, &map);
            if (rc) return rc;
            c = new_launch(key);
            c->decode = false;
            c->pplan = plan;
            c->map = map;
            c->valid = true;
        }
        if (dry) return AFFQMM_OK;
        if (launch_prompt(ws[0].bits, c->pplan.p, c->map, c->pplan.grid, st) != cudaSuccess) return AFFQMM_E_CUDA;
        return AFFQMM_OK;
    }
    // More prompt rows: chunks of up to 128 rows on the tensor-core kernel.
    // The first chunk is the largest: its plan sizes the workspace.
    {
        PromptPlan first;
        rc = plan_prompt(d->sms, count, ws, std::min<int64_t>(M, kPromptRows), &first);
        if (rc) return rc;
        rc = check_workspace(first.ws_bytes, workspace, ws_bytes);
        if (rc || dry) return rc;
    }
    uint8_t* wsb = static_cast<uint8_t*>(workspace);
    for (int64_t m0 = 0; m0 < M; m0 += kPromptRows) {
        const int64_t mc = std::min(kPromptRows, M - m0);
        PromptPlan plan;
        rc = plan_prompt(d->sms, count, ws, mc, &plan);
        if (rc) return rc;
        plan.p.status = reinterpret_cast<uint32_t*>(wsb);
        plan.p.counters = reinterpret_cast<uint32_t*>(wsb + kStatusBytes);
        plan.p.slots = reinterpret_cast<float*>(wsb + kSlotsOffset);
        for (int i = 0; i < count; ++i) plan.p.proj[i].y = ys[i] ? ys[i] + m0 * ws[i].N : nullptr;
        CUtensorMap map;
        rc = make_x_map(x + m0 * K, mc, K, 128, &map);
        if (rc) return rc;
        if (launch_prompt(ws[0].bits, plan.p, map, plan.grid, st) != cudaSuccess) return AFFQMM_E_CUDA;
    }
    return AFFQMM_OK;
}

// The gather from either form of the table: `rows` NULL reads the packed
// blocks of w, else the row-contiguous copy that affqmm_pack_rows made of w.
int embed_impl(const affqmm_weight* w, const void* rows, bool rowcopy, const int32_t* ids, int64_t T, int has_scale,
               uint16_t scale, uint16_t* out, uint32_t* status, void* stream) {
    int rc = check_weight(w);
    if (rc) return rc;
    if (T < 0) return AFFQMM_E_ARG;
    if (T == 0 || w->K == 0) return AFFQMM_OK;
    if (!ids || !out || (rowcopy && !rows)) return AFFQMM_E_NULL;
    if (w->N == 0) return AFFQMM_E_SHAPE;  // no row to gather
    if (!aligned(out, 16) || !aligned(ids, 4) || (status && !aligned(status, 4)) || (rowcopy && !aligned(rows, 256)))
        return AFFQMM_E_ALIGN;
    if (T > ((int64_t)1 << 31) / ((w->K + KBLK - 1) / KBLK)) return AFFQMM_E_SHAPE;
    DeviceInfo* d = nullptr;
    rc = device_info(&d);
    if (rc) return rc;
    if (launch_embed(w->bits, w->group, rowcopy, rowcopy ? rows : w->packed, w->N, w->K, ids, T, has_scale ? 1 : 0,
                     scale, out, status, static_cast<cudaStream_t>(stream)) != cudaSuccess)
        return AFFQMM_E_CUDA;
    return AFFQMM_OK;
}

}  // namespace

extern "C" {

const char* affqmm_strerror(int status) {
    switch (status) {
        case AFFQMM_OK: return "ok";
        case AFFQMM_E_NULL: return "a required pointer is NULL";
        case AFFQMM_E_BITS: return "bits must be 2, 3, 4, 5, 6 or 8";
        case AFFQMM_E_GROUP: return "group must be 32, 64 or 128";
        case AFFQMM_E_SHAPE: return "bad shape (N < 0, K < 0, K not a multiple of group, or too large)";
        case AFFQMM_E_ALIGN: return "a pointer violates its required alignment";
        case AFFQMM_E_M: return "M out of range";
        case AFFQMM_E_WORKSPACE: return "workspace missing or smaller than affqmm_workspace_bytes";
        case AFFQMM_E_TIMEOUT: return "a bounded device wait gave up";
        case AFFQMM_E_CUDA: return "a CUDA call or launch failed";
        case AFFQMM_E_ARG: return "bad argument (count or mismatched stacked weights)";
        case AFFQMM_E_DEVICE: return "the current device is not an sm_103 GPU";
        case AFFQMM_E_SCRATCH:
            return "affqmm_run_noalloc: M > 16, or the work needs more than its 8 MiB built-in scratch";
        default: return "unknown affqmm status";
    }
}

int affqmm_version(void) { return 100; }

int affqmm_packed_bytes(int bits, int group, int64_t N, int64_t K, size_t* bytes) {
    if (!bytes) return AFFQMM_E_NULL;
    if (!valid_bits(bits)) return AFFQMM_E_BITS;
    if (!valid_group(group)) return AFFQMM_E_GROUP;
    if (N < 0 || K < 0 || K % group != 0 || N > (int64_t)1 << 34 || K > (int64_t)1 << 28) return AFFQMM_E_SHAPE;
    const int64_t tiles = (N + TILE_N - 1) / TILE_N;
    const int64_t kb = (K + KBLK - 1) / KBLK;
    if (tiles * kb > ((int64_t)1 << 31) - 1) return AFFQMM_E_SHAPE;
    *bytes = (size_t)tiles * (size_t)kb * (size_t)block_bytes(bits, group);
    return AFFQMM_OK;
}

int affqmm_pack(int bits, int group, int64_t N, int64_t K, const uint8_t* codes, const uint16_t* scales,
                const uint16_t* biases, void* packed, void* stream) {
    size_t bytes = 0;
    int rc = affqmm_packed_bytes(bits, group, N, K, &bytes);
    if (rc) return rc;
    if (bytes == 0) return AFFQMM_OK;
    if (!packed) return AFFQMM_E_NULL;
    if (!aligned(packed, 256)) return AFFQMM_E_ALIGN;
    if (N > 0 && K > 0 && (!codes || !scales || !biases)) return AFFQMM_E_NULL;
    if (launch_pack(bits, group, N, K, codes, scales, biases, packed, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return AFFQMM_E_CUDA;
    return AFFQMM_OK;
}

int affqmm_workspace_bytes(const affqmm_weight* w, int64_t M, size_t* bytes) {
    return affqmm_workspace_bytes_stacked(1, w, M, bytes);
}

int affqmm_workspace_bytes_stacked(int count, const affqmm_weight* ws, int64_t M, size_t* bytes) {
    if (!bytes) return AFFQMM_E_NULL;
    int rc = check_stack(count, ws);
    if (rc) return rc;
    if (M < 0 || M > AFFQMM_MAX_M) return AFFQMM_E_M;
    return workspace_for(count, ws, M, bytes);
}

int affqmm_run(const affqmm_weight* w, const uint16_t* x, int64_t M, uint16_t* y, void* workspace,
               size_t ws_bytes, void* stream) {
    uint16_t* ys[1] = {y};
    return run_impl(1, w, x, M, ys, workspace, ws_bytes, stream);
}

int affqmm_run_exact(const affqmm_weight* w, const uint16_t* x, int64_t M, uint16_t* y, void* workspace,
                     size_t ws_bytes, void* stream) {
    uint16_t* ys[1] = {y};
    Form f;
    f.exact = true;
    return run_impl(1, w, x, M, ys, workspace, ws_bytes, stream, f);
}

int affqmm_run_exact_sums(const affqmm_weight* w, const uint16_t* x, const float* xsums, int64_t M, uint16_t* y,
                          void* workspace, size_t ws_bytes, void* stream) {
    if (M > 0 && w && w->K > 0 && !xsums) return AFFQMM_E_NULL;
    uint16_t* ys[1] = {y};
    Form f;
    f.exact = true;
    f.xsums = xsums;
    return run_impl(1, w, x, M, ys, workspace, ws_bytes, stream, f);
}

int affqmm_run_geglu(const affqmm_weight* w, const uint16_t* x, const float* xsums, int64_t M, int form,
                     uint16_t* h, void* workspace, size_t ws_bytes, void* stream) {
    if (form != AFFQMM_FORM_ROUNDED && form != AFFQMM_FORM_EXACT && form != AFFQMM_FORM_EXACT_SUMS)
        return AFFQMM_E_ARG;
    if (form == AFFQMM_FORM_EXACT_SUMS && M > 0 && w && w->K > 0 && !xsums) return AFFQMM_E_NULL;
    uint16_t* ys[1] = {h};
    Form f;
    f.exact = form != AFFQMM_FORM_ROUNDED;
    f.xsums = form == AFFQMM_FORM_EXACT_SUMS ? xsums : nullptr;
    f.epi = 1;
    return run_impl(1, w, x, M, ys, workspace, ws_bytes, stream, f);
}

int affqmm_run_stacked(int count, const affqmm_weight* ws, const uint16_t* x, int64_t M, uint16_t* const* ys,
                       void* workspace, size_t ws_bytes, void* stream) {
    if (!ys) return AFFQMM_E_NULL;
    return run_impl(count, ws, x, M, ys, workspace, ws_bytes, stream);
}

int affqmm_run_host(const affqmm_weight* w, const uint16_t* x, int64_t M, uint16_t* y, uint16_t* x_dev,
                    uint16_t* y_dev, void* workspace, size_t ws_bytes, void* stream) {
    int rc = check_weight(w);
    if (rc) return rc;
    if (M < 0 || M > AFFQMM_MAX_M) return AFFQMM_E_M;
    if (M == 0 || w->N == 0) return AFFQMM_OK;
    if (!y || !y_dev) return AFFQMM_E_NULL;
    if (w->K > 0 && !x) return AFFQMM_E_NULL;
    uint16_t* ys[1] = {y_dev};
    // every check of the device call (x_dev, y_dev, workspace, device) before anything is enqueued
    rc = run_impl(1, w, x_dev, M, ys, workspace, ws_bytes, stream, Form(), true);
    if (rc) return rc;
    const size_t xbytes = (size_t)M * (size_t)w->K * 2, ybytes = (size_t)M * (size_t)w->N * 2;
    // Page-locked host buffers: the transfers run as kernels chained to the
    // projection (hostio.cu), so that no copy sits between two launches.
    const void* x_gpu = w->K > 0 ? host_on_device(x) : nullptr;
    void* y_gpu = const_cast<void*>(host_on_device(y));
    if ((w->K == 0 || x_gpu) && y_gpu) {
        cudaStream_t st = static_cast<cudaStream_t>(stream);
        if (w->K > 0 && launch_host_upload(x_gpu, x_dev, xbytes, st) != cudaSuccess) return AFFQMM_E_CUDA;
        rc = run_impl(1, w, x_dev, M, ys, workspace, ws_bytes, stream);
        if (rc) return rc;
        if (launch_host_download(y_dev, y_gpu, ybytes, st) != cudaSuccess) return AFFQMM_E_CUDA;
        return AFFQMM_OK;
    }
    CopyHtoDFn htod = copy_htod();
    CopyDtoHFn dtoh = copy_dtoh();
    if (!htod || !dtoh) return AFFQMM_E_CUDA;
    CUstream cs = static_cast<CUstream>(stream);
    if (w->K > 0 && htod(reinterpret_cast<CUdeviceptr>(x_dev), x, xbytes, cs) != CUDA_SUCCESS) return AFFQMM_E_CUDA;
    rc = run_impl(1, w, x_dev, M, ys, workspace, ws_bytes, stream);
    if (rc) return rc;
    if (dtoh(y, reinterpret_cast<CUdeviceptr>(y_dev), ybytes, cs) != CUDA_SUCCESS) return AFFQMM_E_CUDA;
    return AFFQMM_OK;
}

int affqmm_dequant(const affqmm_weight* w, uint16_t* w_out, void* stream) {
    int rc = check_weight(w);
    if (rc) return rc;
    if (w->N == 0 || w->K == 0) return AFFQMM_OK;
    if (!w_out) return AFFQMM_E_NULL;
    if (!aligned(w_out, 2)) return AFFQMM_E_ALIGN;
    if (launch_dequant(w->bits, w->group, w->N, w->K, w->packed, w_out, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return AFFQMM_E_CUDA;
    return AFFQMM_OK;
}

int affqmm_embed_rows(const affqmm_weight* w, const int32_t* ids, int64_t T, int has_scale, uint16_t scale,
                      uint16_t* out, uint32_t* status, void* stream) {
    return embed_impl(w, nullptr, false, ids, T, has_scale, scale, out, status, stream);
}

int affqmm_rows_bytes(int bits, int group, int64_t N, int64_t K, size_t* bytes) {
    size_t packed = 0;
    const int rc = affqmm_packed_bytes(bits, group, N, K, &packed);  // the same argument checks
    if (rc) return rc;
    const int KB = (int)((K + KBLK - 1) / KBLK);
    *bytes = (size_t)N * (size_t)rows_stride(bits, group, KB);
    return AFFQMM_OK;
}

int affqmm_pack_rows(const affqmm_weight* w, void* rows, void* stream) {
    const int rc = check_weight(w);
    if (rc) return rc;
    if (w->N == 0 || w->K == 0) return AFFQMM_OK;
    if (!rows) return AFFQMM_E_NULL;
    if (!aligned(rows, 256)) return AFFQMM_E_ALIGN;
    if (launch_pack_rows(w->bits, w->group, w->packed, w->N, w->K, rows, static_cast<cudaStream_t>(stream)) !=
        cudaSuccess)
        return AFFQMM_E_CUDA;
    return AFFQMM_OK;
}

int affqmm_embed_rows_copy(const affqmm_weight* w, const void* rows, const int32_t* ids, int64_t T, int has_scale,
                           uint16_t scale, uint16_t* out, uint32_t* status, void* stream) {
    return embed_impl(w, rows, true, ids, T, has_scale, scale, out, status, stream);
}

int affqmm_workspace_status(void* workspace, void* stream) {
    if (!workspace) return AFFQMM_E_NULL;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    uint32_t word = 0;
    if (cudaMemcpyAsync(&word, workspace, sizeof word, cudaMemcpyDeviceToHost, st) != cudaSuccess) return AFFQMM_E_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return AFFQMM_E_CUDA;
    if (word == 0) return AFFQMM_OK;
    // A kernel that gave up may have left merge counters behind as well:
    // clear the status word and every counter, the workspace's zeroed prefix.
    if (cudaMemsetAsync(workspace, 0, AFFQMM_WORKSPACE_ZEROED, st) != cudaSuccess) return AFFQMM_E_CUDA;
    if (cudaStreamSynchronize(st) != cudaSuccess) return AFFQMM_E_CUDA;
    return AFFQMM_E_TIMEOUT;
}

int affqmm_test_fault_wait(int64_t cycles) {
    if (cycles < 0) return AFFQMM_E_ARG;
    decode_set_fault_wait(cycles);
    return AFFQMM_OK;
}

}  // extern "C"

// ----------------------------------------------------------------------------
// affqmm_run_noalloc: the decode path (M <= 16) for callers that cannot
// allocate device memory -- a plug-in inside a host engine that owns all of
// the GPU's memory and gives it no allocator, or a latency-critical loop that
// must not call cudaMalloc/cudaFree (which can synchronize the device).  Its
// scratch (status word, merge counters, split-depth partial sums, in the
// workspace layout of affqmm_run) is the file-scope array below, which every
// GPU that loads this library holds until the process exits.  Calls share it:
// calls that overlap on the GPU race on it.

static __device__ __align__(256) uint8_t g_noalloc_scratch[AFFQMM_NOALLOC_SCRATCH_BYTES];

namespace {

// In host code `g_noalloc_scratch` names a host-side stand-in, not device
// memory: kernels get the address that cudaGetSymbolAddress returns for the
// current device, looked up once per device.
// Only a successful lookup is kept: a failed one (for instance, one made
// while the stream was being captured) is tried again on the next call.
struct NoallocScratch {
    void* ptr = nullptr;
    bool ok = false;
};
NoallocScratch g_noalloc[kMaxDevices];
std::mutex g_noalloc_mutex;

int noalloc_scratch(void** out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return AFFQMM_E_CUDA;
    if (dev < 0 || dev >= kMaxDevices) return AFFQMM_E_DEVICE;
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    NoallocScratch& e = g_noalloc[dev];
    if (!e.ok) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr) {
            (void)cudaGetLastError();  // leave no sticky error behind for the caller's next call
            return AFFQMM_E_CUDA;
        }
        e.ptr = p;
        e.ok = true;
    }
    *out = e.ptr;
    return AFFQMM_OK;
}

}  // namespace

extern "C" int affqmm_run_noalloc(const affqmm_weight* w, const uint16_t* x, int64_t M, uint16_t* y,
                                  void* stream) {
    int rc = check_weight(w);
    if (rc) return rc;
    if (M < 0) return AFFQMM_E_M;
    if (M > AFFQMM_NOALLOC_MAX_M) return AFFQMM_E_SCRATCH;
    if (M == 0 || w->N == 0) return AFFQMM_OK;
    if (!y) return AFFQMM_E_NULL;
    if (!aligned(y, 2)) return AFFQMM_E_ALIGN;
    if (w->K > 0) {
        if (!x) return AFFQMM_E_NULL;
        if (!aligned(x, 16)) return AFFQMM_E_ALIGN;
    }
    DeviceInfo* d = nullptr;
    rc = device_info(&d);
    if (rc) return rc;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (w->K == 0) {  // an empty sum: every output is +0
        return cudaMemsetAsync(y, 0, (size_t)M * w->N * 2, st) == cudaSuccess ? AFFQMM_OK : AFFQMM_E_CUDA;
    }
    DecodePlan plan;
    rc = plan_decode(d->sms, d->dec_ctas_per_sm, 1, w, M, &plan);
    if (rc) return rc;
    if (plan.ws_bytes > sizeof(g_noalloc_scratch)) return AFFQMM_E_SCRATCH;
    void* scratch = nullptr;
    rc = noalloc_scratch(&scratch);
    if (rc) return rc;
    // The status word and this call's merge counters (eight per 128-row tile)
    // must start at zero; whatever an earlier call left in them is cleared on
    // the stream, ahead of the kernel.  The partial-sum slots need no clearing.
    const size_t zeroed = kStatusBytes + (size_t)kDecCountersPerTile * (size_t)plan.p.proj[0].tiles * sizeof(uint32_t);
    if (cudaMemsetAsync(scratch, 0, zeroed, st) != cudaSuccess) return AFFQMM_E_CUDA;
    bind_workspace(&plan, scratch);
    plan.p.proj[0].y = y;
    plan.p.x = x;
    CUtensorMap map;
    rc = make_x_map_decode(x, M, w->K, &map);
    if (rc) return rc;
    if (launch_decode(w->bits, w->group, plan.p, map, plan.grid, st) != cudaSuccess) return AFFQMM_E_CUDA;
    return AFFQMM_OK;
}
