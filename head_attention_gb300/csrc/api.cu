// C ABI of libhattn.so: argument validation, kernel dispatch, tensor-map
// construction and caching, and the device error word. See include/hattn.h
// for the contract of every entry point.
#include <cuda.h>
#include <cuda_runtime.h>
#include <nvtx3/nvToolsExt.h>

#include <algorithm>
#include <cmath>
#include <cstring>
#include <mutex>
#include <unordered_map>

#include "internal.h"
#include "ptx.cuh"

namespace hattn {

// First device-side error raised by a kernel of this library on this device.
__device__ int g_device_error = 0;

namespace {

constexpr int kMaxDevices = 64;

int* device_error_ptr()
{
    static int* cache[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return nullptr;
        cache[dev] = static_cast<int*>(p);
    }
    return cache[dev];
}

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
    });
    return fn;
}

// Tensor maps depend only on (pointer, shape, box); cache them so repeated
// calls on the same buffers skip the host-side encode.
struct MapKey {
    const void* base;
    uint64_t dims[4];
    uint32_t box_rows;
    int rank;
    bool operator==(const MapKey& o) const
    {
        return base == o.base && rank == o.rank && box_rows == o.box_rows &&
               std::memcmp(dims, o.dims, sizeof(dims)) == 0;
    }
};
struct MapKeyHash {
    size_t operator()(const MapKey& k) const
    {
        size_t h = std::hash<const void*>()(k.base);
        for (int i = 0; i < 4; ++i) h = h * 1000003u ^ std::hash<uint64_t>()(k.dims[i]);
        return h * 31u + k.box_rows * 7u + k.rank;
    }
};
std::mutex g_map_mu;
std::unordered_map<MapKey, CUtensorMap, MapKeyHash> g_maps;
constexpr size_t kMaxCachedMaps = 4096;

bool cached_map(CUtensorMap* out, const MapKey& key, bool (*make)(CUtensorMap*, const MapKey&))
{
    int dev = 0;
    cudaGetDevice(&dev);
    MapKey k = key;
    k.dims[3] ^= static_cast<uint64_t>(dev) << 48;  // maps are per device
    {
        std::lock_guard<std::mutex> lock(g_map_mu);
        auto it = g_maps.find(k);
        if (it != g_maps.end()) {
            *out = it->second;
            return true;
        }
    }
    if (!make(out, key)) return false;
    std::lock_guard<std::mutex> lock(g_map_mu);
    if (g_maps.size() >= kMaxCachedMaps) g_maps.clear();
    g_maps.emplace(k, *out);
    return true;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// One NVTX range (domain "hattn", named after the entry point) around an entry
// point's host work and launches, so a timeline shows which call enqueued which
// kernels. Without a tool attached a range costs a few nanoseconds.
class Range {
public:
    explicit Range(const char* name)
    {
        static const nvtxDomainHandle_t dom = nvtxDomainCreateA("hattn");
        dom_ = dom;
        nvtxEventAttributes_t a = {};
        a.version = NVTX_VERSION;
        a.size = NVTX_EVENT_ATTRIB_STRUCT_SIZE;
        a.messageType = NVTX_MESSAGE_TYPE_ASCII;
        a.message.ascii = name;
        nvtxDomainRangePushEx(dom_, &a);
    }
    ~Range() { nvtxDomainRangePop(dom_); }
    Range(const Range&) = delete;
    Range& operator=(const Range&) = delete;

private:
    nvtxDomainHandle_t dom_;
};

int from_cuda(cudaError_t e) { return e == cudaSuccess ? HATTN_OK : HATTN_ECUDA; }

bool make_bnhd_uncached(CUtensorMap* map, const MapKey& k)
{
    // dims = {d, h, n, B}
    const uint64_t d = k.dims[0], h = k.dims[1], n = k.dims[2], B = k.dims[3];
    const uint64_t dims[4] = {d, h, n, B};
    const uint64_t strides[3] = {d * 2, h * d * 2, n * h * d * 2};
    const uint32_t box[4] = {64, 1, k.box_rows, 1};
    return encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, k.base, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

bool make_2d_uncached(CUtensorMap* map, const MapKey& k)
{
    // dims = {cols, rows}, box = {64, box_rows}
    const uint64_t dims[2] = {k.dims[0], k.dims[1]};
    const uint64_t strides[1] = {k.dims[0] * 2};
    const uint32_t box[2] = {64, k.box_rows};
    return encode_tmap(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, k.base, dims, strides, box,
                       CU_TENSOR_MAP_SWIZZLE_128B);
}

// Row-major bf16 [rows][cols] matrix, boxes of 64 columns x box_rows rows.
bool make_2d_map(CUtensorMap* map, const void* base, int rows, int cols, int box_rows)
{
    MapKey k{base, {(uint64_t)cols, (uint64_t)rows, 0, 0}, (uint32_t)box_rows, 2};
    return cached_map(map, k, make_2d_uncached);
}

}  // namespace

bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base,
                 const uint64_t* dims, const uint64_t* strides_bytes, const uint32_t* box,
                 CUtensorMapSwizzle swizzle)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    cuuint64_t gdim[5], gstride[4];
    cuuint32_t bdim[5], estride[5];
    for (int i = 0; i < rank; ++i) {
        gdim[i] = dims[i];
        bdim[i] = box[i];
        estride[i] = 1;
    }
    for (int i = 0; i < rank - 1; ++i) gstride[i] = strides_bytes[i];
    CUresult r = fn(map, dtype, rank, const_cast<void*>(base), gdim, gstride, bdim, estride,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool make_bnhd_map(CUtensorMap* map, const void* base, int B, int n, int h, int d, int box_rows)
{
    MapKey k{base, {(uint64_t)d, (uint64_t)h, (uint64_t)n, (uint64_t)B}, (uint32_t)box_rows, 4};
    return cached_map(map, k, make_bnhd_uncached);
}

namespace {

int validate_attn(const void* q, const void* k, const void* v, void* out, int dtype, int B, int h,
                  int n_q, int n_k, int d_k, int d_v, float scale, int mask_kind,
                  const int32_t* key_lens)
{
    if (!q || !k || !v || !out) return HATTN_EINVAL;
    if (dtype != HATTN_F32 && dtype != HATTN_BF16) return HATTN_EINVAL;
    if (B <= 0 || h <= 0 || n_q <= 0 || n_k <= 0 || d_k <= 0 || d_v <= 0) return HATTN_EINVAL;
    if (mask_kind & ~(HATTN_MASK_CAUSAL | HATTN_MASK_KEY_PADDING)) return HATTN_EINVAL;
    if ((mask_kind & HATTN_MASK_CAUSAL) && n_q != n_k) return HATTN_EINVAL;
    if ((mask_kind & HATTN_MASK_KEY_PADDING) && !key_lens) return HATTN_EINVAL;
    if (!std::isfinite(scale)) return HATTN_EINVAL;
    if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out)) return HATTN_EINVAL;
    const size_t esz = dtype == HATTN_F32 ? 4 : 2;
    if ((d_k * esz) % 16 != 0 || (d_v * esz) % 16 != 0) return HATTN_EINVAL;
    if (dtype == HATTN_F32 && (d_k > 128 || d_v > 128)) return HATTN_EUNSUPPORTED;
    if (dtype == HATTN_BF16 && (d_k > 256 || d_v > 256)) return HATTN_EUNSUPPORTED;
    return HATTN_OK;
}

int run_attn(const AttnArgs& a)
{
    if (attn_short_supported(a)) {
        AttnMaps m;
        if (!make_bnhd_map(&m.q, a.q, a.B, a.n_q, a.h, a.d_k, 128) ||
            !make_bnhd_map(&m.k, a.k, a.B, a.n_k, a.h, a.d_k, 128) ||
            !make_bnhd_map(&m.v, a.v, a.B, a.n_k, a.h, a.d_v, 128) ||
            !make_bnhd_map(&m.o, a.out, a.B, a.n_q, a.h, a.d_v, 128))
            return HATTN_ECUDA;
        return from_cuda(launch_attn_short(a, m));
    }
    if (attn_tc_supported(a)) {
        AttnMaps m;
        if (!make_bnhd_map(&m.q, a.q, a.B, a.n_q, a.h, a.d_k, 128) ||
            !make_bnhd_map(&m.k, a.k, a.B, a.n_k, a.h, a.d_k, 128) ||
            !make_bnhd_map(&m.v, a.v, a.B, a.n_k, a.h, a.d_v, 128))
            return HATTN_ECUDA;
        return from_cuda(launch_attn_tc(a, m));
    }
    if (a.h > 65535 || a.B > 65535) return HATTN_EUNSUPPORTED;
    return from_cuda(launch_attn_simt(a));
}

size_t align256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

struct MhaLayout {
    size_t q, k, v, a, total;
};

bool mha_layout(int B, int n_q, int n_k, int h, int d_k, int d_v, MhaLayout* L)
{
    if (B <= 0 || n_q <= 0 || n_k <= 0 || h <= 0 || d_k <= 0 || d_v <= 0) return false;
    const size_t q = (size_t)B * n_q * h * d_k * 2, k = (size_t)B * n_k * h * d_k * 2;
    const size_t v = (size_t)B * n_k * h * d_v * 2, a = (size_t)B * n_q * h * d_v * 2;
    L->q = 0;
    L->k = L->q + align256(q);
    L->v = L->k + align256(k);
    L->a = L->v + align256(v);
    L->total = L->a + align256(a);
    return true;
}

}  // namespace
}  // namespace hattn

using namespace hattn;

extern "C" {

int attn_fwd(const void* q, const void* k, const void* v, void* out, int dtype, int B, int h,
             int n_q, int n_k, int d_k, int d_v, float scale, int mask_kind,
             const int32_t* key_lens, hattn_stream_t stream)
{
    const Range range("attn_fwd");
    int rc = validate_attn(q, k, v, out, dtype, B, h, n_q, n_k, d_k, d_v, scale, mask_kind,
                           key_lens);
    if (rc != HATTN_OK) return rc;
    AttnArgs a{q, k, v, out, dtype, B, h, n_q, n_k, d_k, d_v, scale, mask_kind,
               (mask_kind & HATTN_MASK_KEY_PADDING) ? key_lens : nullptr,
               reinterpret_cast<cudaStream_t>(stream), device_error_ptr()};
    if (!a.err_word) return HATTN_ECUDA;
    return run_attn(a);
}

size_t mha_workspace_bytes(int dtype, int B, int n_q, int n_k, int d_model, int h, int d_k,
                           int d_v)
{
    MhaLayout L;
    if (dtype != HATTN_BF16 || d_model <= 0 || !mha_layout(B, n_q, n_k, h, d_k, d_v, &L)) return 0;
    return L.total;
}

int mha_fwd(const void* x_q, const void* x_kv, const void* Wq, const void* Wk, const void* Wv,
            const void* Wo, const float* gamma, const float* beta, float eps, void* y, int dtype,
            int B, int n_q, int n_k, int d_model, int h, int d_k, int d_v, int mask_kind,
            const int32_t* key_lens, void* workspace, size_t ws_bytes, hattn_stream_t stream)
{
    const Range range("mha_fwd");
    if (!x_q || !x_kv || !Wq || !Wk || !Wv || !Wo || !gamma || !beta || !y) return HATTN_EINVAL;
    if (dtype != HATTN_BF16) return dtype == HATTN_F32 ? HATTN_EUNSUPPORTED : HATTN_EINVAL;
    if (B <= 0 || n_q <= 0 || n_k <= 0 || d_model <= 0 || h <= 0 || d_k <= 0 || d_v <= 0)
        return HATTN_EINVAL;
    if (mask_kind & ~(HATTN_MASK_CAUSAL | HATTN_MASK_KEY_PADDING)) return HATTN_EINVAL;
    if ((mask_kind & HATTN_MASK_CAUSAL) && n_q != n_k) return HATTN_EINVAL;
    if ((mask_kind & HATTN_MASK_KEY_PADDING) && !key_lens) return HATTN_EINVAL;
    if (!(eps > 0.0f) || !std::isfinite(eps)) return HATTN_EINVAL;
    const void* ptrs[] = {x_q, x_kv, Wq, Wk, Wv, Wo, gamma, beta, y};
    for (const void* p : ptrs)
        if (!aligned16(p)) return HATTN_EINVAL;
    if (d_k != d_v || (d_k != 64 && d_k != 128)) return HATTN_EUNSUPPORTED;
    if (d_model % 64 != 0 || d_model > 512 || (h * d_k) % 64 != 0) return HATTN_EUNSUPPORTED;
    MhaLayout L;
    if (!mha_layout(B, n_q, n_k, h, d_k, d_v, &L)) return HATTN_EINVAL;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || ws_bytes < L.total)
        return HATTN_EWORKSPACE;
    int* err = device_error_ptr();
    if (!err) return HATTN_ECUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    char* ws = static_cast<char*>(workspace);
    void* Q = ws + L.q;
    void* K = ws + L.k;
    void* V = ws + L.v;
    void* A = ws + L.a;
    const int Mq = B * n_q, Mk = B * n_k, hdk = h * d_k, hdv = h * d_v;

    ProjProblem pr[3];
    const void* xs[3] = {x_q, x_kv, x_kv};
    const void* ws3[3] = {Wq, Wk, Wv};
    void* outs[3] = {Q, K, V};
    const int Ms[3] = {Mq, Mk, Mk};
    const int Ns[3] = {hdk, hdk, hdv};
    for (int i = 0; i < 3; ++i) {
        if (!make_2d_map(&pr[i].a, xs[i], Ms[i], d_model, 128) ||
            !make_2d_map(&pr[i].w, ws3[i], d_model, Ns[i], 64) ||
            !make_2d_map(&pr[i].cmap, outs[i], Ms[i], Ns[i], 32))
            return HATTN_ECUDA;
        pr[i].c = outs[i];
        pr[i].M = Ms[i];
        pr[i].N = Ns[i];
        pr[i].K = d_model;
    }
    int rc = from_cuda(launch_proj_gemm(pr, 3, st, err));
    if (rc != HATTN_OK) return rc;

    AttnArgs a{Q, K, V, A, HATTN_BF16, B, h, n_q, n_k, d_k, d_v,
               1.0f / std::sqrt(static_cast<float>(d_k)), mask_kind,
               (mask_kind & HATTN_MASK_KEY_PADDING) ? key_lens : nullptr, st, err};
    rc = run_attn(a);
    if (rc != HATTN_OK) return rc;

    OutProjLnArgs o;
    if (!make_2d_map(&o.a, A, Mq, hdv, 128) || !make_2d_map(&o.wo, Wo, hdv, d_model, 64) ||
        !make_2d_map(&o.xmap, x_q, Mq, d_model, 128) || !make_2d_map(&o.ymap, y, Mq, d_model, 32))
        return HATTN_ECUDA;
    o.x = x_q;
    o.gamma = gamma;
    o.beta = beta;
    o.eps = eps;
    o.y = y;
    o.M = Mq;
    o.N = d_model;
    o.K = hdv;
    return from_cuda(launch_outproj_ln(o, st, err));
}

}  // extern "C"

namespace hattn {
namespace {

// The static scratch of mha_fwd_noalloc: Q, K, V and the concatenated heads of
// one call, laid out exactly as mha_fwd lays out its workspace.
static __device__ __align__(256) unsigned char g_noalloc_scratch[HATTN_NOALLOC_SCRATCH_BYTES];

// Device address of g_noalloc_scratch on the current device, looked up once per
// device with that device current (host code only has a stand-in for the name).
void* noalloc_scratch_ptr()
{
    static void* cache[kMaxDevices] = {};
    static std::mutex mu;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(mu);
    if (!cache[dev]) {
        void* p = nullptr;
        if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess) return nullptr;
        cache[dev] = p;
    }
    return cache[dev];
}

}  // namespace
}  // namespace hattn

extern "C" {

int mha_fwd_noalloc(const void* x_q, const void* x_kv, const void* Wq, const void* Wk,
                    const void* Wv, const void* Wo, const float* gamma, const float* beta,
                    float eps, void* y, int dtype, int B, int n_q, int n_k, int d_model, int h,
                    int d_k, int d_v, int mask_kind, const int32_t* key_lens,
                    hattn_stream_t stream)
{
    const Range range("mha_fwd_noalloc");
    // Missing or misaligned buffers and a wrong dtype are reported as such whatever
    // the problem size; then an oversized request is rejected before any CUDA call.
    const void* bufs[] = {x_q, x_kv, Wq, Wk, Wv, Wo, gamma, beta, y};
    for (const void* p : bufs)
        if (!p || !aligned16(p)) return HATTN_EINVAL;
    if (dtype != HATTN_BF16) return dtype == HATTN_F32 ? HATTN_EUNSUPPORTED : HATTN_EINVAL;
    const size_t need = mha_workspace_bytes(dtype, B, n_q, n_k, d_model, h, d_k, d_v);
    if (need > HATTN_NOALLOC_SCRATCH_BYTES) return HATTN_ESCRATCH;
    if (need == 0) {
        // Bad sizes or dtype: let mha_fwd's own checks report them (no workspace needed).
        return mha_fwd(x_q, x_kv, Wq, Wk, Wv, Wo, gamma, beta, eps, y, dtype, B, n_q, n_k,
                       d_model, h, d_k, d_v, mask_kind, key_lens, nullptr, 0, stream);
    }
    void* scratch = noalloc_scratch_ptr();
    if (!scratch) return HATTN_ECUDA;
    return mha_fwd(x_q, x_kv, Wq, Wk, Wv, Wo, gamma, beta, eps, y, dtype, B, n_q, n_k, d_model,
                   h, d_k, d_v, mask_kind, key_lens, scratch, HATTN_NOALLOC_SCRATCH_BYTES, stream);
}

int attn_fwd_lse(const void* q, const void* k, const void* v, void* out, float* lse, int dtype,
                 int B, int h, int n_q, int n_k, int d_k, int d_v, float scale, int mask_kind,
                 const int32_t* key_lens, hattn_stream_t stream)
{
    const Range range("attn_fwd_lse");
    if (!lse || !aligned16(lse)) return HATTN_EINVAL;
    int rc = validate_attn(q, k, v, out, dtype, B, h, n_q, n_k, d_k, d_v, scale, mask_kind,
                           key_lens);
    if (rc != HATTN_OK) return rc;
    AttnArgs a{q, k, v, out, dtype, B, h, n_q, n_k, d_k, d_v, scale, mask_kind,
               (mask_kind & HATTN_MASK_KEY_PADDING) ? key_lens : nullptr,
               reinterpret_cast<cudaStream_t>(stream), device_error_ptr(), lse};
    if (!a.err_word) return HATTN_ECUDA;
    return run_attn(a);
}

size_t attn_bwd_workspace_bytes(int B, int h, int n_q)
{
    if (B <= 0 || h <= 0 || n_q <= 0) return 0;
    const size_t nqp = ((size_t)n_q + 127) / 128 * 128;
    return 2 * sizeof(float) * (size_t)B * h * nqp;  // dsum and lse2, each a multiple of 512 B
}

int attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
             const float* lse, void* dq, void* dk, void* dv, int dtype, int B, int h, int n_q,
             int n_k, int d_k, int d_v, float scale, int mask_kind, const int32_t* key_lens,
             void* workspace, size_t ws_bytes, hattn_stream_t stream)
{
    const Range range("attn_bwd");
    if (!dout || !lse || !dq || !dk || !dv) return HATTN_EINVAL;
    const void* ptrs[] = {dout, lse, dq, dk, dv};
    for (const void* ptr : ptrs)
        if (!aligned16(ptr)) return HATTN_EINVAL;
    int rc = validate_attn(q, k, v, const_cast<void*>(out), dtype, B, h, n_q, n_k, d_k, d_v,
                           scale, mask_kind, key_lens);
    if (rc != HATTN_OK) return rc;
    if (h > 65535 || B > 65535) return HATTN_EUNSUPPORTED;
    const size_t need = attn_bwd_workspace_bytes(B, h, n_q);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || ws_bytes < need)
        return HATTN_EWORKSPACE;
    int* err = device_error_ptr();
    if (!err) return HATTN_ECUDA;
    const size_t nqp = ((size_t)n_q + 127) / 128 * 128;
    float* dsum = static_cast<float*>(workspace);
    float* lse2 = dsum + (size_t)B * h * nqp;
    AttnBwdArgs a{q, k, v, out, dout, lse, dq, dk, dv, dsum, lse2, dtype,
                  B, h, n_q, n_k, d_k, d_v, scale, mask_kind,
                  (mask_kind & HATTN_MASK_KEY_PADDING) ? key_lens : nullptr,
                  reinterpret_cast<cudaStream_t>(stream), err};
    rc = from_cuda(launch_attn_bwd_prep(a));
    if (rc != HATTN_OK) return rc;
    if (attn_bwd_tc_supported(a)) {
        AttnMaps m;
        CUtensorMap g;
        if (!make_bnhd_map(&m.q, q, B, n_q, h, d_k, 128) || !make_bnhd_map(&m.k, k, B, n_k, h, d_k, 128) ||
            !make_bnhd_map(&m.v, v, B, n_k, h, d_v, 128) || !make_bnhd_map(&g, dout, B, n_q, h, d_v, 128))
            return HATTN_ECUDA;
        return from_cuda(launch_attn_bwd_tc(a, m, g));
    }
    return from_cuda(launch_attn_bwd_simt(a));
}

size_t attn_decode_workspace_bytes(int B, int h, int n_max, int d)
{
    if (B <= 0 || h <= 0 || n_max <= 0 || (d != 64 && d != 128 && d != 256)) return 0;
    int splits = 0, chunk = 0;
    decode_split_plan(B, h, n_max, &splits, &chunk);
    return sizeof(float) * (size_t)B * h * splits * (d + 2);
}

int attn_decode_fwd(const void* q, const void* k_cache, const void* v_cache, void* out, int dtype,
                    int B, int h, int n_max, int d, float scale, const int32_t* kv_lens,
                    void* workspace, size_t ws_bytes, hattn_stream_t stream)
{
    const Range range("attn_decode_fwd");
    if (!q || !k_cache || !v_cache || !out || !kv_lens) return HATTN_EINVAL;
    if (dtype != HATTN_BF16) return dtype == HATTN_F32 ? HATTN_EUNSUPPORTED : HATTN_EINVAL;
    if (B <= 0 || h <= 0 || n_max <= 0 || d <= 0 || !std::isfinite(scale)) return HATTN_EINVAL;
    if (B > 65535 || h > 65535) return HATTN_EUNSUPPORTED;
    if (d != 64 && d != 128 && d != 256) return HATTN_EUNSUPPORTED;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out))
        return HATTN_EINVAL;
    const size_t need = attn_decode_workspace_bytes(B, h, n_max, d);
    if (!workspace || !aligned16(workspace) || ws_bytes < need) return HATTN_EWORKSPACE;
    int* err = device_error_ptr();
    if (!err) return HATTN_ECUDA;
    DecodeLaunch a{q, k_cache, v_cache, out, kv_lens, workspace, B, h, n_max, d, 0, 0, scale,
                   reinterpret_cast<cudaStream_t>(stream), err};
    decode_split_plan(B, h, n_max, &a.splits, &a.chunk);
    return from_cuda(launch_attn_decode(a));
}

int pos_encoding_fwd(const void* emb, void* out, int dtype, int B, int n, int d_model,
                     float emb_scale, int pos0, hattn_stream_t stream)
{
    const Range range("pos_encoding_fwd");
    if (!out || (dtype != HATTN_F32 && dtype != HATTN_BF16)) return HATTN_EINVAL;
    if (B <= 0 || n <= 0 || d_model <= 0 || (d_model & 1) || pos0 < 0) return HATTN_EINVAL;
    if ((long long)pos0 + n > (1LL << 24) || !std::isfinite(emb_scale)) return HATTN_EINVAL;
    if ((reinterpret_cast<uintptr_t>(out) & 7u) || (reinterpret_cast<uintptr_t>(emb) & 7u))
        return HATTN_EINVAL;
    int* err = device_error_ptr();
    if (!err) return HATTN_ECUDA;
    return from_cuda(launch_pos_encoding(emb, out, dtype, B, n, d_model, emb_scale, pos0, err,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

}  // extern "C"

namespace hattn {
namespace {

bool ffn_shapes_ok(int M, int d_model, int d_ff)
{
    return M > 0 && d_model > 0 && d_ff > 0;
}

int ffn_supported(int d_model, int d_ff)
{
    return (d_model % 64 == 0 && d_model <= 512 && d_ff % 64 == 0) ? HATTN_OK : HATTN_EUNSUPPORTED;
}

}  // namespace
}  // namespace hattn

extern "C" {

size_t ffn_workspace_bytes(int dtype, int M, int d_model, int d_ff)
{
    if (dtype != HATTN_BF16 || !ffn_shapes_ok(M, d_model, d_ff)) return 0;
    return align256((size_t)M * d_ff * 2);
}

int ffn_fwd(const void* x, const void* W1, const float* b1, const void* W2, const float* b2,
            const float* gamma, const float* beta, float eps, void* y, int dtype, int M,
            int d_model, int d_ff, void* workspace, size_t ws_bytes, hattn_stream_t stream)
{
    const Range range("ffn_fwd");
    if (!x || !W1 || !W2 || !gamma || !beta || !y) return HATTN_EINVAL;
    if (dtype != HATTN_BF16) return dtype == HATTN_F32 ? HATTN_EUNSUPPORTED : HATTN_EINVAL;
    if (!ffn_shapes_ok(M, d_model, d_ff)) return HATTN_EINVAL;
    if (!(eps > 0.0f) || !std::isfinite(eps)) return HATTN_EINVAL;
    const void* ptrs[] = {x, W1, W2, gamma, beta, y};
    for (const void* p : ptrs)
        if (!aligned16(p)) return HATTN_EINVAL;
    if ((b1 && !aligned16(b1)) || (b2 && !aligned16(b2))) return HATTN_EINVAL;
    if (x == y) return HATTN_EINVAL;
    int rc = ffn_supported(d_model, d_ff);
    if (rc != HATTN_OK) return rc;
    const size_t need = ffn_workspace_bytes(dtype, M, d_model, d_ff);
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || ws_bytes < need)
        return HATTN_EWORKSPACE;
    int* err = device_error_ptr();
    if (!err) return HATTN_ECUDA;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    void* H = workspace;
    // H = max(0, x W1 + b1)
    ProjProblem pr;
    if (!make_2d_map(&pr.a, x, M, d_model, 128) || !make_2d_map(&pr.w, W1, d_model, d_ff, 64) ||
        !make_2d_map(&pr.cmap, H, M, d_ff, 32))
        return HATTN_ECUDA;
    pr.c = H;
    pr.M = M;
    pr.N = d_ff;
    pr.K = d_model;
    pr.bias = b1;
    pr.relu = true;
    rc = from_cuda(launch_proj_gemm(&pr, 1, st, err));
    if (rc != HATTN_OK) return rc;
    // y = LN(x + H W2 + b2)
    OutProjLnArgs o;
    if (!make_2d_map(&o.a, H, M, d_ff, 128) || !make_2d_map(&o.wo, W2, d_ff, d_model, 64) ||
        !make_2d_map(&o.xmap, x, M, d_model, 128) || !make_2d_map(&o.ymap, y, M, d_model, 32))
        return HATTN_ECUDA;
    o.x = x;
    o.gamma = gamma;
    o.beta = beta;
    o.eps = eps;
    o.y = y;
    o.M = M;
    o.N = d_model;
    o.K = d_ff;
    o.bias = b2;
    return from_cuda(launch_outproj_ln(o, st, err));
}

size_t encoder_layer_workspace_bytes(int dtype, int B, int n, int d_model, int h, int d_k,
                                     int d_ff)
{
    const size_t mha = mha_workspace_bytes(dtype, B, n, n, d_model, h, d_k, d_k);
    const size_t ffn = ((long long)B * n > 0x7fffffffLL) ? 0 : ffn_workspace_bytes(dtype, B * n, d_model, d_ff);
    if (mha == 0 || ffn == 0) return 0;
    return std::max(mha, ffn) + align256((size_t)B * n * d_model * 2);
}

int encoder_layer_fwd(const void* x, const hattn_mha_weights* attn, const hattn_ffn_weights* ffn,
                      float eps, void* y, int dtype, int B, int n, int d_model, int h, int d_k,
                      int d_ff, const int32_t* key_lens, void* workspace, size_t ws_bytes,
                      hattn_stream_t stream)
{
    const Range range("encoder_layer_fwd");
    if (!x || !attn || !ffn || !y) return HATTN_EINVAL;
    if (B <= 0 || n <= 0 || (long long)B * n > 0x7fffffffLL) return HATTN_EINVAL;
    const size_t need = encoder_layer_workspace_bytes(dtype, B, n, d_model, h, d_k, d_ff);
    if (need == 0) return dtype == HATTN_F32 ? HATTN_EUNSUPPORTED : HATTN_EINVAL;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || ws_bytes < need)
        return HATTN_EWORKSPACE;
    const size_t scratch = need - align256((size_t)B * n * d_model * 2);
    void* y1 = static_cast<char*>(workspace) + scratch;
    const int mask = key_lens ? HATTN_MASK_KEY_PADDING : HATTN_MASK_NONE;
    int rc = mha_fwd(x, x, attn->Wq, attn->Wk, attn->Wv, attn->Wo, attn->gamma, attn->beta, eps,
                     y1, dtype, B, n, n, d_model, h, d_k, d_k, mask, key_lens, workspace, scratch,
                     stream);
    if (rc != HATTN_OK) return rc;
    return ffn_fwd(y1, ffn->W1, ffn->b1, ffn->W2, ffn->b2, ffn->gamma, ffn->beta, eps, y, dtype,
                   B * n, d_model, d_ff, workspace, scratch, stream);
}

size_t decoder_layer_workspace_bytes(int dtype, int B, int n_tgt, int n_src, int d_model, int h,
                                     int d_k, int d_ff)
{
    const size_t self = mha_workspace_bytes(dtype, B, n_tgt, n_tgt, d_model, h, d_k, d_k);
    const size_t cross = mha_workspace_bytes(dtype, B, n_tgt, n_src, d_model, h, d_k, d_k);
    const size_t ffn =
        ((long long)B * n_tgt > 0x7fffffffLL) ? 0 : ffn_workspace_bytes(dtype, B * n_tgt, d_model, d_ff);
    if (self == 0 || cross == 0 || ffn == 0) return 0;
    return std::max(std::max(self, cross), ffn) + 2 * align256((size_t)B * n_tgt * d_model * 2);
}

int decoder_layer_fwd(const void* x, const void* memory, const hattn_mha_weights* self_attn,
                      const hattn_mha_weights* cross_attn, const hattn_ffn_weights* ffn, float eps,
                      void* y, int dtype, int B, int n_tgt, int n_src, int d_model, int h,
                      int d_k, int d_ff, const int32_t* src_lens, void* workspace,
                      size_t ws_bytes, hattn_stream_t stream)
{
    const Range range("decoder_layer_fwd");
    if (!x || !memory || !self_attn || !cross_attn || !ffn || !y) return HATTN_EINVAL;
    if (B <= 0 || n_tgt <= 0 || n_src <= 0 || (long long)B * n_tgt > 0x7fffffffLL)
        return HATTN_EINVAL;
    const size_t need =
        decoder_layer_workspace_bytes(dtype, B, n_tgt, n_src, d_model, h, d_k, d_ff);
    if (need == 0) return dtype == HATTN_F32 ? HATTN_EUNSUPPORTED : HATTN_EINVAL;
    if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u) != 0 || ws_bytes < need)
        return HATTN_EWORKSPACE;
    const size_t act = align256((size_t)B * n_tgt * d_model * 2);
    const size_t scratch = need - 2 * act;
    void* y1 = static_cast<char*>(workspace) + scratch;
    void* y2 = static_cast<char*>(y1) + act;
    int rc = mha_fwd(x, x, self_attn->Wq, self_attn->Wk, self_attn->Wv, self_attn->Wo,
                     self_attn->gamma, self_attn->beta, eps, y1, dtype, B, n_tgt, n_tgt, d_model,
                     h, d_k, d_k, HATTN_MASK_CAUSAL, nullptr, workspace, scratch, stream);
    if (rc != HATTN_OK) return rc;
    rc = mha_fwd(y1, memory, cross_attn->Wq, cross_attn->Wk, cross_attn->Wv, cross_attn->Wo,
                 cross_attn->gamma, cross_attn->beta, eps, y2, dtype, B, n_tgt, n_src, d_model, h,
                 d_k, d_k, src_lens ? HATTN_MASK_KEY_PADDING : HATTN_MASK_NONE, src_lens,
                 workspace, scratch, stream);
    if (rc != HATTN_OK) return rc;
    return ffn_fwd(y2, ffn->W1, ffn->b1, ffn->W2, ffn->b2, ffn->gamma, ffn->beta, eps, y, dtype,
                   B * n_tgt, d_model, d_ff, workspace, scratch, stream);
}

const char* hattn_status_str(int status)
{
    switch (status) {
    case HATTN_OK: return "ok";
    case HATTN_EINVAL: return "invalid argument";
    case HATTN_EUNSUPPORTED: return "unsupported configuration";
    case HATTN_ECUDA: return "CUDA error";
    case HATTN_ETIMEOUT: return "device pipeline wait timed out";
    case HATTN_EKEYLEN: return "key length outside [1, n_k]";
    case HATTN_EWORKSPACE: return "workspace missing, misaligned or too small";
    case HATTN_ESCRATCH: return "problem needs more than the 32 MiB static scratch of mha_fwd_noalloc";
    default: return "unknown status";
    }
}

int hattn_check_device_error(hattn_stream_t stream)
{
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return HATTN_ECUDA;
    int value = 0;
    if (cudaMemcpyFromSymbol(&value, g_device_error, sizeof(int)) != cudaSuccess)
        return HATTN_ECUDA;
    if (value != 0) {
        const int zero = 0;
        if (cudaMemcpyToSymbol(g_device_error, &zero, sizeof(int)) != cudaSuccess)
            return HATTN_ECUDA;
    }
    return value;
}

int hattn_version(void) { return 100; }

}  // extern "C"

namespace hattn {
namespace {

// One thread waits on an mbarrier that nothing arrives on, through the same
// bounded wait every pipeline of this library uses; when the wait gives up it
// raises HATTN_ETIMEOUT in the device error word and the kernel returns.
__global__ void wait_timeout_selftest_kernel(int* err_word)
{
    __shared__ __align__(8) uint64_t bar;
    if (threadIdx.x != 0) return;
    const uint32_t b = smem_u32(&bar);
    mbar_init(b, 1);
    fence_barrier_init();
    if (!mbar_wait(b, 0)) raise_device_error(err_word, HATTN_ETIMEOUT);
}

}  // namespace
}  // namespace hattn

extern "C" {

int hattn_selftest_wait_timeout(hattn_stream_t stream)
{
    const hattn::Range range("hattn_selftest_wait_timeout");
    int* err = hattn::device_error_ptr();
    if (!err) return HATTN_ECUDA;
    hattn::wait_timeout_selftest_kernel<<<1, 32, 0, reinterpret_cast<cudaStream_t>(stream)>>>(err);
    return hattn::from_cuda(cudaGetLastError());
}

}  // extern "C"
