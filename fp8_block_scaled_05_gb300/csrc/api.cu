// C-ABI entry points (include/fp8bs.h): argument validation, per-device
// state, TMA descriptor cache and kernel dispatch.  Host code only.
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_runtime.h>

#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <atomic>
#include <mutex>
#include <unordered_map>

#include "fp8bs.h"
#include "internal.h"

namespace fp8bs {
namespace {

// First error recorded by any kernel on this device (0 = none).
__device__ int g_device_status;

constexpr int kMaxDevices = 64;
std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

fp8_status cuda_status(cudaError_t e) { return e == cudaSuccess ? FP8_OK : FP8_ERR_CUDA; }

// Current device, checked to be sm_103, with its SM count and status word.
fp8_status current_device(DeviceInfo** out) {
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return FP8_ERR_ARCH;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DeviceInfo& d = g_dev[dev];
    if (d.device < 0) {
        int major = 0, minor = 0, sms = 0, smem = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&smem, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) {
            cudaGetLastError();
            return FP8_ERR_ARCH;
        }
        if (major != 10 || minor != 3) return FP8_ERR_ARCH;
        void* sym = nullptr;
        if (cudaGetSymbolAddress(&sym, g_device_status) != cudaSuccess) {
            cudaGetLastError();
            return FP8_ERR_CUDA;
        }
        if (cudaMemset(sym, 0, sizeof(int)) != cudaSuccess) return FP8_ERR_CUDA;
        if (!g_encode) {
            cudaDriverEntryPointQueryResult q;
            void* fn = nullptr;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
                    cudaSuccess ||
                q != cudaDriverEntryPointSuccess || !fn) {
                cudaGetLastError();
                return FP8_ERR_CUDA;
            }
            g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
        }
        d.sm_count = sms;
        d.max_smem_optin = smem;
        d.status = static_cast<int*>(sym);
        d.device = dev;
    }
    *out = &d;
    return FP8_OK;
}

// ------------------------------------------------------------ TMA descriptors
struct TmKey {
    uint64_t ptr, d0, d1, pitch;
    uint32_t b0, b1;
    int dtype, swizzle;
    bool operator==(const TmKey& o) const { return std::memcmp(this, &o, sizeof(TmKey)) == 0; }
};
struct TmKeyHash {
    size_t operator()(const TmKey& k) const {
        uint64_t h = 1469598103934665603ull;
        const unsigned char* p = reinterpret_cast<const unsigned char*>(&k);
        for (size_t i = 0; i < sizeof(TmKey); ++i) h = (h ^ p[i]) * 1099511628211ull;
        return (size_t)h;
    }
};
std::mutex g_tm_mu;
std::unordered_map<TmKey, CUtensorMap, TmKeyHash> g_tm_cache;

// 2-D row-major tensor [d1 rows][d0 elements], row pitch in bytes, box
// {b0, b1}.  Descriptors are cached by all of these (a descriptor depends on
// nothing else) and copied out under the lock, so a later eviction of the
// cache cannot invalidate a caller's copy.
fp8_status tensor_map(const void* ptr, CUtensorMapDataType dtype, uint64_t d0, uint64_t d1, uint64_t pitch_bytes,
                      uint32_t b0, uint32_t b1, CUtensorMapSwizzle swz, CUtensorMap* out) {
    TmKey key;
    std::memset(&key, 0, sizeof(key));
    key.ptr = reinterpret_cast<uint64_t>(ptr);
    key.d0 = d0;
    key.d1 = d1;
    key.pitch = pitch_bytes;
    key.b0 = b0;
    key.b1 = b1;
    key.dtype = (int)dtype;
    key.swizzle = (int)swz;
    std::lock_guard<std::mutex> lk(g_tm_mu);
    auto it = g_tm_cache.find(key);
    if (it != g_tm_cache.end()) {
        *out = it->second;
        return FP8_OK;
    }
    if (g_tm_cache.size() > 4096) g_tm_cache.clear();
    CUtensorMap m;
    const cuuint64_t dims[2] = {d0, d1};
    const cuuint64_t strides[1] = {pitch_bytes};
    const cuuint32_t box[2] = {b0, b1};
    const cuuint32_t estr[2] = {1, 1};
    CUresult r = g_encode(&m, dtype, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, swz, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return FP8_ERR_CUDA;
    g_tm_cache.emplace(key, m);
    *out = m;
    return FP8_OK;
}

fp8_status check_mode(int mode) { return (mode == FP8_SCALE_FP32_AMAX || mode == FP8_SCALE_POW2) ? FP8_OK : FP8_ERR_SCALE_MODE; }

constexpr uint32_t kKnownFlags = FP8_GEMM_SCALES_POW2 | FP8_GEMM_SCALES_E8 | FP8_GEMM_PATH_MASK;

// Path of a dense GEMM: the one forced by the flags, else the skinny kernel
// for M <= 128, else the MX kernel when the caller promises power-of-two
// scales and the promote kernel otherwise.  From 129 rows the skinny kernel
// runs two token chunks per weight tile and the large-M kernels, each tile
// split along K over the SMs, measured faster (M = 256: 33 -> 25 us at
// N 6144, K 4096; 48 -> 36 us at N 4096, K 14336); up to 128 rows the skinny
// kernel is as fast or faster (M <= 64: 17 against 25 us, 23 against 37 us).
uint32_t plan_path(int64_t M, int64_t K, uint32_t flags) {
    const uint32_t forced = flags & FP8_GEMM_PATH_MASK;
    if (forced != FP8_GEMM_PATH_AUTO) return forced;
    if (flags & FP8_GEMM_SCALES_E8) return FP8_GEMM_PATH_MX;   // byte scales: the MX kernel reads them
    if (M <= kSkinnyAutoMaxM && K <= 128 * 1024) return FP8_GEMM_PATH_SKINNY;
    return (flags & FP8_GEMM_SCALES_POW2) ? FP8_GEMM_PATH_MX : FP8_GEMM_PATH_PROMOTE;
}

// Path of a grouped GEMM: forced, else MX for power-of-two scales, else promote.
uint32_t grouped_path(uint32_t flags) {
    const uint32_t forced = flags & FP8_GEMM_PATH_MASK;
    if (forced != FP8_GEMM_PATH_AUTO) return forced;
    if (flags & FP8_GEMM_SCALES_E8) return FP8_GEMM_PATH_MX;
    return (flags & FP8_GEMM_SCALES_POW2) ? FP8_GEMM_PATH_MX : FP8_GEMM_PATH_PROMOTE;
}

// Shared validation of the GEMM operands (both forms).
fp8_status check_gemm_common(const void* qa, int64_t lda, const float* sa, int64_t ldsa, const void* qb,
                             const float* sb, const void* c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                             uint32_t flags) {
    if (M < 0 || N <= 0 || K <= 0 || (N % 128) || (K % 128)) return FP8_ERR_SHAPE;
    if (M > INT32_MAX / 2 || N > (1ll << 24) || K > (1ll << 24)) return FP8_ERR_SHAPE;
    if (flags & ~kKnownFlags) return FP8_ERR_SCALE_MODE;
    const uint32_t path = flags & FP8_GEMM_PATH_MASK;
    if (path > FP8_GEMM_PATH_SKINNY) return FP8_ERR_SCALE_MODE;
    if (path == FP8_GEMM_PATH_MX && !(flags & (FP8_GEMM_SCALES_POW2 | FP8_GEMM_SCALES_E8))) return FP8_ERR_SCALE_MODE;
    if (M == 0) return FP8_OK;
    if (!qa || !sa || !qb || !sb || !c) return FP8_ERR_NULL;
    if (lda < K || ldc < N || ldsa < M) return FP8_ERR_SHAPE;
    if ((lda % 16) || (ldsa % 4) || (ldc % 8)) return FP8_ERR_ALIGN;
    if (!aligned16(qa) || !aligned16(sa) || !aligned16(qb) || !aligned16(sb) || !aligned16(c)) return FP8_ERR_ALIGN;
    return FP8_OK;
}

}  // namespace

// Tile width of the promote kernel.  128 gives four TMEM accumulator buffers
// (more slack between the tensor core and the promotion warps), 256 halves
// the operand traffic per FLOP.  FP8BS_PROMOTE_BN=128|256 overrides the
// choice (for tuning).
int promote_tile_n(int64_t M, int64_t N, int64_t K, int32_t G) {
    (void)M;
    (void)K;
    (void)G;
    static int forced = [] {
        const char* e = std::getenv("FP8BS_PROMOTE_BN");
        if (!e) return 0;
        const int v = std::atoi(e);
        return (v == 128 || v == 256) ? v : 0;
    }();
    if (forced) return forced;
    return (N % 256 == 0) ? 256 : 128;
}

// Failure-path test hook (fp8_debug_inject): read by every GEMM call.
namespace {
std::atomic<uint64_t> g_inject_wait_ns{0};
std::atomic<int32_t> g_inject_skip{0};
}  // namespace

void fault_injection(uint64_t* wait_ns, int32_t* skip_first_load) {
    *wait_ns = g_inject_wait_ns.load(std::memory_order_relaxed);
    *skip_first_load = g_inject_skip.load(std::memory_order_relaxed);
}

}  // namespace fp8bs

using namespace fp8bs;

extern "C" {

const char* fp8_status_string(fp8_status st) {
    switch (st) {
        case FP8_OK: return "FP8_OK";
        case FP8_ERR_NULL: return "FP8_ERR_NULL: a required pointer is NULL";
        case FP8_ERR_SHAPE: return "FP8_ERR_SHAPE: sizes out of range or leading dimension too small";
        case FP8_ERR_ALIGN: return "FP8_ERR_ALIGN: pointer or row pitch not 16-byte aligned";
        case FP8_ERR_SCALE_MODE: return "FP8_ERR_SCALE_MODE: unknown scale mode or flags";
        case FP8_ERR_WORKSPACE: return "FP8_ERR_WORKSPACE: workspace missing or too small";
        case FP8_ERR_ARCH: return "FP8_ERR_ARCH: no sm_103 CUDA device is current";
        case FP8_ERR_CUDA: return "FP8_ERR_CUDA: a CUDA call failed";
        case FP8_ERR_TIMEOUT: return "FP8_ERR_TIMEOUT: a kernel wait ran out of time";
        case FP8_ERR_NOT_IMPLEMENTED: return "FP8_ERR_NOT_IMPLEMENTED: path not built";
    }
    return "unknown fp8_status";
}

fp8_status fp8_quant_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq, float* s,
                               int64_t lds, fp8_scale_mode mode, fp8_stream_t stream) {
    if (fp8_status e = check_mode(mode)) return e;
    if (M < 0 || K <= 0 || (K % 128) || M > (1ll << 31) - 1 || K > (1ll << 26)) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (!x || !q || !s) return FP8_ERR_NULL;
    if (ldx < K || ldq < K || lds < M) return FP8_ERR_SHAPE;
    if ((ldx % 8) || (ldq % 16) || (lds % 4) || !aligned16(x) || !aligned16(q) || !aligned16(s)) return FP8_ERR_ALIGN;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    return cuda_status(launch_quant_act_1x128(x, M, K, ldx, q, ldq, s, lds, mode == FP8_SCALE_POW2,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

fp8_status fp8_quant_act_weight(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* qa, int64_t ldqa,
                                float* sa, int64_t ldsa, const void* w, int64_t N, int64_t ldw, uint8_t* qw,
                                int64_t ldqw, float* sw, fp8_scale_mode mode, fp8_stream_t stream) {
    if (fp8_status e = check_mode(mode)) return e;
    if (M < 0 || K <= 0 || (K % 128) || M > (1ll << 31) - 1 || K > (1ll << 26)) return FP8_ERR_SHAPE;
    if (N <= 0 || (N % 128) || N / 128 > 65535) return FP8_ERR_SHAPE;
    const int64_t blocks = (N / 128) * (K / 128) + ((M + 15) / 16) * ((K / 128 + 7) / 8);
    if (blocks > INT32_MAX) return FP8_ERR_SHAPE;
    if (!w || !qw || !sw) return FP8_ERR_NULL;
    if (M > 0 && (!x || !qa || !sa)) return FP8_ERR_NULL;
    if (ldw < K || ldqw < K) return FP8_ERR_SHAPE;
    if (M > 0 && (ldx < K || ldqa < K || ldsa < M)) return FP8_ERR_SHAPE;
    if ((ldw % 8) || (ldqw % 16) || !aligned16(w) || !aligned16(qw) || (reinterpret_cast<uintptr_t>(sw) % 4))
        return FP8_ERR_ALIGN;
    if (M > 0 && ((ldx % 8) || (ldqa % 16) || (ldsa % 4) || !aligned16(x) || !aligned16(qa) || !aligned16(sa)))
        return FP8_ERR_ALIGN;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    return cuda_status(launch_quant_act_weight(x, M, K, ldx, qa, ldqa, sa, ldsa, w, N, ldw, qw, ldqw, sw,
                                               mode == FP8_SCALE_POW2, reinterpret_cast<cudaStream_t>(stream)));
}

fp8_status fp8_quant_act_1x128_e8(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq,
                                  uint8_t* s, int64_t lds, fp8_stream_t stream) {
    if (M < 0 || K <= 0 || (K % 128) || M > (1ll << 31) - 1 || K > (1ll << 26)) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (!x || !q || !s) return FP8_ERR_NULL;
    if (ldx < K || ldq < K || lds < M) return FP8_ERR_SHAPE;
    if ((ldx % 8) || (ldq % 16) || (lds % 4) || !aligned16(x) || !aligned16(q)) return FP8_ERR_ALIGN;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    return cuda_status(launch_quant_act_1x128(x, M, K, ldx, q, ldq, nullptr, lds, true,
                                              reinterpret_cast<cudaStream_t>(stream), s));
}

fp8_status fp8_quant_weight_128x128_e8(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q, int64_t ldq,
                                       uint8_t* s, fp8_stream_t stream) {
    if (N <= 0 || K <= 0 || (N % 128) || (K % 128) || N / 128 > 65535 || K > (1ll << 30)) return FP8_ERR_SHAPE;
    if (!w || !q || !s) return FP8_ERR_NULL;
    if (ldw < K || ldq < K) return FP8_ERR_SHAPE;
    if ((ldw % 8) || (ldq % 16) || !aligned16(w) || !aligned16(q)) return FP8_ERR_ALIGN;   // s: bytes, any address
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    return cuda_status(launch_quant_weight_128x128(w, N, K, ldw, q, ldq, nullptr, true,
                                                   reinterpret_cast<cudaStream_t>(stream), s));
}

fp8_status fp8_quant_weight_128x128(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q, int64_t ldq,
                                    float* s, fp8_scale_mode mode, fp8_stream_t stream) {
    if (fp8_status e = check_mode(mode)) return e;
    if (N <= 0 || K <= 0 || (N % 128) || (K % 128) || N / 128 > 65535 || K > (1ll << 30)) return FP8_ERR_SHAPE;
    if (!w || !q || !s) return FP8_ERR_NULL;
    if (ldw < K || ldq < K) return FP8_ERR_SHAPE;
    if ((ldw % 8) || (ldq % 16) || !aligned16(w) || !aligned16(q) || (reinterpret_cast<uintptr_t>(s) % 4))
        return FP8_ERR_ALIGN;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    return cuda_status(launch_quant_weight_128x128(w, N, K, ldw, q, ldq, s, mode == FP8_SCALE_POW2,
                                                   reinterpret_cast<cudaStream_t>(stream)));
}

fp8_status fp8_quant_act_128x1(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* qt, int64_t ldqt,
                               float* st, int64_t ldst, uint8_t* q, int64_t ldq, float* s, int64_t lds,
                               fp8_scale_mode mode, fp8_stream_t stream) {
    if (fp8_status e = check_mode(mode)) return e;
    if (M < 0 || K <= 0 || (K % 128) || (M + 127) / 128 > 65535 || K > (1ll << 30)) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (!x || !qt || !st) return FP8_ERR_NULL;
    if ((q == nullptr) != (s == nullptr)) return FP8_ERR_NULL;   // the 1x128 outputs come as a pair
    const int64_t Mp = (M + 127) / 128 * 128;                    // tokens padded to whole 128x1 blocks
    if (ldx < K || ldqt < Mp || ldst < K) return FP8_ERR_SHAPE;
    if ((ldx % 8) || (ldqt % 16) || (ldst % 4) || !aligned16(x) || !aligned16(qt) || !aligned16(st))
        return FP8_ERR_ALIGN;
    if (q != nullptr) {
        if (ldq < K || lds < M) return FP8_ERR_SHAPE;
        if ((ldq % 16) || (lds % 4) || !aligned16(q) || !aligned16(s)) return FP8_ERR_ALIGN;
    }
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    return cuda_status(launch_quant_act_128x1(x, M, K, ldx, qt, ldqt, st, ldst, q, ldq, s, lds,
                                              mode == FP8_SCALE_POW2, reinterpret_cast<cudaStream_t>(stream)));
}

fp8_status fp8_quant_act_128x1_grouped(const void* x, int64_t T, int64_t K, int64_t ldx, const int32_t* offsets,
                                      int32_t G, uint8_t* qt, int64_t ldqt, float* st, int64_t ldst,
                                      fp8_scale_mode mode, fp8_stream_t stream) {
    if (fp8_status e = check_mode(mode)) return e;
    if (T < 0 || K <= 0 || (K % 128) || G < 1 || G > kMaxGroupedQuantExperts || T > INT32_MAX / 2 ||
        K > (1ll << 30))
        return FP8_ERR_SHAPE;
    const int64_t nbmax = grouped_token_blocks(T, G);
    if (nbmax > 65535) return FP8_ERR_SHAPE;
    if (T == 0) return FP8_OK;
    if (!x || !offsets || !qt || !st) return FP8_ERR_NULL;
    if (ldx < K || ldqt < 128 * nbmax || ldst < K) return FP8_ERR_SHAPE;
    if ((ldx % 8) || (ldqt % 16) || (ldst % 4) || !aligned16(x) || !aligned16(qt) || !aligned16(st) ||
        (reinterpret_cast<uintptr_t>(offsets) % 4))
        return FP8_ERR_ALIGN;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    return cuda_status(launch_quant_act_128x1_grouped(x, T, K, ldx, offsets, G, qt, ldqt, st, ldst,
                                                      mode == FP8_SCALE_POW2, reinterpret_cast<cudaStream_t>(stream)));
}

fp8_status fp8_quant_weight_128x128_t(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q, int64_t ldq,
                                      float* s, uint8_t* qt, int64_t ldqt, float* st, fp8_scale_mode mode,
                                      fp8_stream_t stream) {
    if (fp8_status e = check_mode(mode)) return e;
    if (N <= 0 || K <= 0 || (N % 128) || (K % 128) || N / 128 > 65535 || K > (1ll << 30)) return FP8_ERR_SHAPE;
    if (!w || !qt || !st) return FP8_ERR_NULL;
    if ((q == nullptr) != (s == nullptr)) return FP8_ERR_NULL;   // W's own codes come as a pair
    if (ldw < K || ldqt < N) return FP8_ERR_SHAPE;
    if ((ldw % 8) || (ldqt % 16) || !aligned16(w) || !aligned16(qt) || !aligned16(st)) return FP8_ERR_ALIGN;
    if (q != nullptr) {
        if (ldq < K) return FP8_ERR_SHAPE;
        if ((ldq % 16) || !aligned16(q) || !aligned16(s)) return FP8_ERR_ALIGN;
    }
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    return cuda_status(launch_quant_weight_128x128_t(w, N, K, ldw, q, ldq, s, qt, ldqt, st, mode == FP8_SCALE_POW2,
                                                     reinterpret_cast<cudaStream_t>(stream)));
}

fp8_status fp8_quant_per_tensor(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq,
                                float* scale_amax, fp8_scale_mode mode, fp8_stream_t stream) {
    if (fp8_status e = check_mode(mode)) return e;
    if (M < 0 || K <= 0 || (K % 8) || M > (1ll << 40) || K > (1ll << 40)) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (!x || !q || !scale_amax) return FP8_ERR_NULL;
    if (ldx < K || ldq < K) return FP8_ERR_SHAPE;
    if ((ldx % 8) || (ldq % 16) || !aligned16(x) || !aligned16(q) || (reinterpret_cast<uintptr_t>(scale_amax) % 8))
        return FP8_ERR_ALIGN;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    return cuda_status(launch_quant_per_tensor(x, M, K, ldx, q, ldq, scale_amax, mode == FP8_SCALE_POW2, d->sm_count,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

fp8_status fp8_quant_with_scale(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq,
                                const float* scale, fp8_stream_t stream) {
    if (M < 0 || K <= 0 || (K % 8) || M > (1ll << 40) || K > (1ll << 40)) return FP8_ERR_SHAPE;
    if (M == 0) return FP8_OK;
    if (!x || !q || !scale) return FP8_ERR_NULL;
    if (ldx < K || ldq < K) return FP8_ERR_SHAPE;
    if ((ldx % 8) || (ldq % 16) || !aligned16(x) || !aligned16(q) || (reinterpret_cast<uintptr_t>(scale) % 4))
        return FP8_ERR_ALIGN;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    return cuda_status(launch_cast_with_scale(x, M, K, ldx, q, ldq, scale, d->sm_count,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

fp8_status fp8_kv_cache_append(const void* k_new, const void* v_new, const float* sk, const float* sv,
                               const int32_t* seq_lens, uint8_t* k_cache, uint8_t* v_cache, int64_t B, int64_t Hkv,
                               int64_t T, int64_t D, fp8_stream_t stream) {
    if (B < 0 || Hkv <= 0 || T <= 0 || D != 128 || B > 65535 || Hkv > 65535 || T > (1 << 24)) return FP8_ERR_SHAPE;
    if (B * Hkv > INT32_MAX) return FP8_ERR_SHAPE;
    if (B == 0) return FP8_OK;
    if (!k_new || !v_new || !sk || !sv || !seq_lens || !k_cache || !v_cache) return FP8_ERR_NULL;
    if (!aligned16(k_new) || !aligned16(v_new) || !aligned16(k_cache) || !aligned16(v_cache) ||
        (reinterpret_cast<uintptr_t>(seq_lens) % 4) || (reinterpret_cast<uintptr_t>(sk) % 4) ||
        (reinterpret_cast<uintptr_t>(sv) % 4))
        return FP8_ERR_ALIGN;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    return cuda_status(launch_kv_append(k_new, v_new, sk, sv, seq_lens, k_cache, v_cache, (int)B, (int)Hkv, (int)T,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

size_t fp8_decode_attention_workspace_size(int64_t B, int64_t Hq, int64_t T) {
    if (B <= 0 || Hq <= 0 || T <= 0 || B > 65535 || Hq > 4096 || T > (1 << 24)) return 0;
    return attn_workspace_bytes((int)B, (int)Hq, (int)T);
}

fp8_status fp8_decode_attention(const uint8_t* q, const float* sq, const uint8_t* k_cache, const float* sk,
                                const uint8_t* v_cache, const float* sv, const int32_t* seq_lens, int64_t B,
                                int64_t Hq, int64_t Hkv, int64_t T, int64_t D, void* out, void* workspace,
                                size_t ws_bytes, fp8_stream_t stream) {
    if (B < 0 || Hq <= 0 || Hkv <= 0 || T <= 0 || D != 128) return FP8_ERR_SHAPE;
    if (Hq % Hkv) return FP8_ERR_SHAPE;
    const int64_t G = Hq / Hkv;
    if (G != 1 && G != 2 && G != 4 && G != 8) return FP8_ERR_SHAPE;
    if (B > 65535 || Hkv > 65535 || T > (1 << 24) || Hq > 4096) return FP8_ERR_SHAPE;
    if (B == 0) return FP8_OK;
    if (!q || !sq || !k_cache || !sk || !v_cache || !sv || !seq_lens || !out) return FP8_ERR_NULL;
    if (!aligned16(q) || !aligned16(k_cache) || !aligned16(v_cache) || !aligned16(out) ||
        (reinterpret_cast<uintptr_t>(seq_lens) % 4) || (reinterpret_cast<uintptr_t>(sq) % 4) ||
        (reinterpret_cast<uintptr_t>(sk) % 4) || (reinterpret_cast<uintptr_t>(sv) % 4))
        return FP8_ERR_ALIGN;
    const size_t need = attn_workspace_bytes((int)B, (int)Hq, (int)T);
    if (need > 0 && (!workspace || ws_bytes < need || !aligned16(workspace))) return FP8_ERR_WORKSPACE;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    return cuda_status(launch_decode_attention(q, sq, k_cache, sk, v_cache, sv, seq_lens, (int)B, (int)Hq, (int)Hkv,
                                               (int)T, workspace, static_cast<uint16_t*>(out),
                                               reinterpret_cast<cudaStream_t>(stream)));
}

uint32_t fp8_gemm_plan(int64_t M, int64_t N, int64_t K, uint32_t flags, int32_t* splits) {
    const uint32_t path = plan_path(M, K, flags);
    int32_t sp = 1;
    if (path == FP8_GEMM_PATH_SKINNY) {
        int sms = 152;
        DeviceInfo* d;
        if (current_device(&d) == FP8_OK) sms = d->sm_count;
        sp = skinny_splits(M, N, K, sms);
    }
    if (splits) *splits = sp;
    return path;
}

// The largest need of the paths these sizes may take (automatic or forced):
// the large-M kernels' K split and, up to 256 rows, the skinny kernel's
// partials, so that one size query serves every flag.
size_t fp8_gemm_workspace_size(int64_t M, int64_t N, int64_t K, int32_t G) {
    if (G != 1 || M <= 0 || N <= 0 || K <= 0) return 0;
    int sms = 152;
    DeviceInfo* d;
    if (current_device(&d) == FP8_OK) sms = d->sm_count;
    size_t need = promote_workspace_bytes(M, N, K, sms);
    if (M <= 256) {
        const size_t s = skinny_workspace_bytes(M, N, K, skinny_splits(M, N, K, sms));
        if (s > need) need = s;
    }
    return need;
}

fp8_status fp8_blockscaled_gemm(const uint8_t* qa, int64_t lda, const float* sa, int64_t ldsa, const uint8_t* qb,
                                int64_t ldb, const float* sb, void* c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                uint32_t flags, void* workspace, size_t ws_bytes, fp8_stream_t stream) {
    if (fp8_status e = check_gemm_common(qa, lda, sa, ldsa, qb, sb, c, ldc, M, N, K, flags)) return e;
    if (M == 0) return FP8_OK;
    if (ldb < K) return FP8_ERR_SHAPE;
    if (ldb % 16) return FP8_ERR_ALIGN;
    const uint32_t path = plan_path(M, K, flags);
    if ((flags & FP8_GEMM_SCALES_E8) && path != FP8_GEMM_PATH_MX) return FP8_ERR_NOT_IMPLEMENTED;
    if (path == FP8_GEMM_PATH_SKINNY && (M > 256 || K / 128 > 1024)) return FP8_ERR_SHAPE;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;

    GemmArgs a{};
    fault_injection(&a.wait_ns, &a.skip_first_load);
    a.sa = sa;
    a.ldsa = ldsa;
    a.sb = sb;
    a.c = c;
    a.ldc = ldc;
    a.M = M;
    a.N = N;
    a.K = K;
    a.offsets = nullptr;
    a.G = 1;
    a.status = d->status;
    a.sm_count = d->sm_count;
    a.splits = 1;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);

    if (path == FP8_GEMM_PATH_SKINNY) {
        const int nt = skinny_tile_n(M);
        a.splits = skinny_splits(M, N, K, d->sm_count);
        const size_t need = skinny_workspace_bytes(M, N, K, a.splits);
        if (need > 0 && (!workspace || ws_bytes < need || !aligned16(workspace))) return FP8_ERR_WORKSPACE;
        a.workspace = workspace;
        a.ws_bytes = ws_bytes;
        a.qb = qb;
        a.ldb = ldb;
        if (fp8_status e = tensor_map(qa, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, lda, 128, nt,
                                      CU_TENSOR_MAP_SWIZZLE_128B, &a.tm_a))
            return e;
        if (fp8_status e = tensor_map(qb, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, N, ldb, 128, 128,
                                      CU_TENSOR_MAP_SWIZZLE_128B, &a.tm_b))
            return e;
        return cuda_status(launch_gemm_skinny(a, st));
    }
    const bool mx = path == FP8_GEMM_PATH_MX;
    a.scales_e8 = (flags & FP8_GEMM_SCALES_E8) ? 1 : 0;
    a.bn = mx ? kMxTileN : promote_tile_n(M, N, K, 1);
    if (workspace && aligned16(workspace)) {
        // optional: lets the kernel split its last wave of tiles
        a.workspace = workspace;
        a.ws_bytes = ws_bytes;
    }
    if (fp8_status e = tensor_map(c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M, ldc * 2, 32, 32,
                                  CU_TENSOR_MAP_SWIZZLE_64B, &a.tm_c))
        return e;
    if (fp8_status e = tensor_map(qa, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, lda, 128, 128,
                                  CU_TENSOR_MAP_SWIZZLE_128B, &a.tm_a))
        return e;
    if (fp8_status e = tensor_map(qb, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, N, ldb, 128, (uint32_t)a.bn,
                                  CU_TENSOR_MAP_SWIZZLE_128B, &a.tm_b))
        return e;
    return cuda_status(mx ? launch_gemm_mx(a, st) : launch_gemm_promote(a, st));
}

fp8_status fp8_blockscaled_gemm_wgrad(const uint8_t* qa, int64_t lda, const float* sa, int64_t ldsa,
                                      const uint8_t* qb, int64_t ldb, const float* sb, int64_t ldsb, void* c,
                                      int64_t ldc, int64_t M, int64_t N, int64_t K, uint32_t flags, void* workspace,
                                      size_t ws_bytes, fp8_stream_t stream) {
    if (flags & FP8_GEMM_SCALES_E8) return FP8_ERR_NOT_IMPLEMENTED;   // fp32 scales only
    if (fp8_status e = check_gemm_common(qa, lda, sa, ldsa, qb, sb, c, ldc, M, N, K, flags)) return e;
    const uint32_t forced = flags & FP8_GEMM_PATH_MASK;
    if (forced == FP8_GEMM_PATH_SKINNY) return FP8_ERR_NOT_IMPLEMENTED;
    const bool mx = forced == FP8_GEMM_PATH_MX || (forced == FP8_GEMM_PATH_AUTO && (flags & FP8_GEMM_SCALES_POW2));
    if (M == 0) return FP8_OK;
    if (ldb < K || ldsb < N) return FP8_ERR_SHAPE;
    if ((ldb % 16) || (ldsb % 4)) return FP8_ERR_ALIGN;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;

    GemmArgs a{};
    fault_injection(&a.wait_ns, &a.skip_first_load);
    a.sa = sa;
    a.ldsa = ldsa;
    a.sb = sb;
    a.ldsb = ldsb;
    a.c = c;
    a.ldc = ldc;
    a.M = M;
    a.N = N;
    a.K = K;
    a.offsets = nullptr;
    a.G = 1;
    a.status = d->status;
    a.sm_count = d->sm_count;
    a.splits = 1;
    a.bn = mx ? kMxTileN : promote_tile_n(M, N, K, 1);
    if (workspace && aligned16(workspace)) {
        a.workspace = workspace;
        a.ws_bytes = ws_bytes;
    }
    if (fp8_status e = tensor_map(c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M, ldc * 2, 32, 32,
                                  CU_TENSOR_MAP_SWIZZLE_64B, &a.tm_c))
        return e;
    if (fp8_status e = tensor_map(qa, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, lda, 128, 128,
                                  CU_TENSOR_MAP_SWIZZLE_128B, &a.tm_a))
        return e;
    if (fp8_status e = tensor_map(qb, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, N, ldb, 128, (uint32_t)a.bn,
                                  CU_TENSOR_MAP_SWIZZLE_128B, &a.tm_b))
        return e;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return cuda_status(mx ? launch_gemm_mx(a, st) : launch_gemm_promote(a, st));
}

fp8_status fp8_blockscaled_grouped_gemm_wgrad(const uint8_t* qa, int64_t lda, const float* sa, int64_t ldsa,
                                              const uint8_t* qb, int64_t ldb, const float* sb, int64_t ldsb,
                                              const int32_t* offsets, int32_t G, int64_t T, void* c, int64_t ldc,
                                              int64_t M, int64_t N, uint32_t flags, fp8_stream_t stream) {
    if (flags & FP8_GEMM_SCALES_E8) return FP8_ERR_NOT_IMPLEMENTED;   // fp32 scales only
    if (flags & ~kKnownFlags) return FP8_ERR_SCALE_MODE;
    const uint32_t path = flags & FP8_GEMM_PATH_MASK;
    if (path > FP8_GEMM_PATH_SKINNY) return FP8_ERR_SCALE_MODE;
    if (path == FP8_GEMM_PATH_MX && !(flags & FP8_GEMM_SCALES_POW2)) return FP8_ERR_SCALE_MODE;
    if (path == FP8_GEMM_PATH_SKINNY) return FP8_ERR_NOT_IMPLEMENTED;
    // power-of-two scales accumulate in TMEM with hardware scale factors (MX)
    const bool mx = path == FP8_GEMM_PATH_MX || (path == FP8_GEMM_PATH_AUTO && (flags & FP8_GEMM_SCALES_POW2));
    if (M < 0 || N < 0 || (M % 128) || (N % 128) || M > (1ll << 24) || N > (1ll << 24)) return FP8_ERR_SHAPE;
    if (G < 1 || G > kMaxGroupedQuantExperts || T < 0 || T > INT32_MAX / 2) return FP8_ERR_SHAPE;
    if ((int64_t)G * M > INT32_MAX) return FP8_ERR_SHAPE;
    if (M == 0 || N == 0) return FP8_OK;
    const int64_t kcap = 128 * grouped_token_blocks(T, G);   // padded token slots the quantiser may fill
    if (!qa || !sa || !qb || !sb || !c || !offsets) return FP8_ERR_NULL;
    if (lda < kcap || ldb < kcap || ldsa < M || ldsb < N || ldc < N) return FP8_ERR_SHAPE;
    if ((lda % 16) || (ldb % 16) || (ldsa % 4) || (ldsb % 4) || (ldc % 8)) return FP8_ERR_ALIGN;
    if (!aligned16(qa) || !aligned16(sa) || !aligned16(qb) || !aligned16(sb) || !aligned16(c) ||
        (reinterpret_cast<uintptr_t>(offsets) % 4))
        return FP8_ERR_ALIGN;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    GemmArgs a{};
    fault_injection(&a.wait_ns, &a.skip_first_load);
    a.sa = sa;
    a.ldsa = ldsa;
    a.sb = sb;
    a.ldsb = ldsb;
    a.c = c;
    a.ldc = ldc;
    a.M = M;
    a.N = N;
    a.K = kcap;
    a.offsets = offsets;
    a.G = G;
    a.kgroup = 1;
    a.kg_tokens = T;
    a.status = d->status;
    a.sm_count = d->sm_count;
    a.splits = 1;
    a.bn = mx ? kMxTileN : promote_tile_n(M, N, kcap, G);
    if (fp8_status e = tensor_map(c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, (uint64_t)G * M, ldc * 2, 32, 32,
                                  CU_TENSOR_MAP_SWIZZLE_64B, &a.tm_c))
        return e;
    if (fp8_status e = tensor_map(qa, CU_TENSOR_MAP_DATA_TYPE_UINT8, kcap, M, lda, 128, 128,
                                  CU_TENSOR_MAP_SWIZZLE_128B, &a.tm_a))
        return e;
    if (fp8_status e = tensor_map(qb, CU_TENSOR_MAP_DATA_TYPE_UINT8, kcap, N, ldb, 128, (uint32_t)a.bn,
                                  CU_TENSOR_MAP_SWIZZLE_128B, &a.tm_b))
        return e;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return cuda_status(mx ? launch_gemm_mx(a, st) : launch_gemm_promote(a, st));
}

fp8_status fp8_tensorscaled_gemm(const uint8_t* qa, int64_t lda, const float* sa, const uint8_t* qb, int64_t ldb,
                                 const float* sb, void* c, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                 uint32_t flags, void* workspace, size_t ws_bytes, fp8_stream_t stream) {
    if (flags & FP8_GEMM_SCALES_E8) return FP8_ERR_SCALE_MODE;   // one fp32 scale per operand
    // the block-scaled validation with the one-scale pointers standing in for
    // the scale arrays (ldsa = M keeps its pitch rule satisfied)
    if (fp8_status e = check_gemm_common(qa, lda, sa, M > 0 ? ((M + 3) / 4) * 4 : 0, qb, sb, c, ldc, M, N, K,
                                         flags | FP8_GEMM_SCALES_POW2))
        return e;
    const uint32_t forced = flags & FP8_GEMM_PATH_MASK;
    if (forced == FP8_GEMM_PATH_PROMOTE || forced == FP8_GEMM_PATH_SKINNY) return FP8_ERR_NOT_IMPLEMENTED;
    if (M == 0) return FP8_OK;
    if (ldb < K) return FP8_ERR_SHAPE;
    if (ldb % 16) return FP8_ERR_ALIGN;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;

    GemmArgs a{};
    fault_injection(&a.wait_ns, &a.skip_first_load);
    a.per_tensor = 1;
    a.sa = sa;
    a.sb = sb;
    a.c = c;
    a.ldc = ldc;
    a.M = M;
    a.N = N;
    a.K = K;
    a.offsets = nullptr;
    a.G = 1;
    a.status = d->status;
    a.sm_count = d->sm_count;
    a.splits = 1;
    a.bn = kMxTileN;
    if (workspace && aligned16(workspace)) {
        a.workspace = workspace;
        a.ws_bytes = ws_bytes;
    }
    if (fp8_status e = tensor_map(c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M, ldc * 2, 32, 32,
                                  CU_TENSOR_MAP_SWIZZLE_64B, &a.tm_c))
        return e;
    if (fp8_status e = tensor_map(qa, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, lda, 128, 128,
                                  CU_TENSOR_MAP_SWIZZLE_128B, &a.tm_a))
        return e;
    if (fp8_status e = tensor_map(qb, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, N, ldb, 128, (uint32_t)a.bn,
                                  CU_TENSOR_MAP_SWIZZLE_128B, &a.tm_b))
        return e;
    return cuda_status(launch_gemm_mx(a, reinterpret_cast<cudaStream_t>(stream)));
}

fp8_status fp8_blockscaled_gemm_quant(const uint8_t* qa, int64_t lda, const float* sa, int64_t ldsa, const uint8_t* qb,
                                      int64_t ldb, const float* sb, void* c, int64_t ldc, uint8_t* qc, int64_t ldqc,
                                      float* sc, int64_t ldsc, int64_t M, int64_t N, int64_t K, uint32_t flags,
                                      fp8_scale_mode out_mode, void* workspace, size_t ws_bytes,
                                      fp8_stream_t stream) {
    if (flags & FP8_GEMM_SCALES_E8) return FP8_ERR_NOT_IMPLEMENTED;   // fp32 scales only
    if (fp8_status e = check_mode(out_mode)) return e;
    // c is optional here: validate with the codes standing in for it
    if (fp8_status e = check_gemm_common(qa, lda, sa, ldsa, qb, sb, c ? c : static_cast<const void*>(qc),
                                         c ? ldc : N, M, N, K, flags))
        return e;
    // large-M kernels only: MX for power-of-two scales (its epilogue warps have
    // the time), promote otherwise
    const uint32_t forced = flags & FP8_GEMM_PATH_MASK;
    if (forced == FP8_GEMM_PATH_SKINNY) return FP8_ERR_NOT_IMPLEMENTED;
    const bool mx = forced == FP8_GEMM_PATH_MX || (forced == FP8_GEMM_PATH_AUTO && (flags & FP8_GEMM_SCALES_POW2));
    if (M == 0) return FP8_OK;
    if (!qc || !sc) return FP8_ERR_NULL;
    if (ldb < K || ldqc < N || ldsc < M) return FP8_ERR_SHAPE;
    if ((ldb % 16) || (ldqc % 16) || (ldsc % 4) || !aligned16(qc) || !aligned16(sc)) return FP8_ERR_ALIGN;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    GemmArgs a{};
    fault_injection(&a.wait_ns, &a.skip_first_load);
    a.sa = sa;
    a.ldsa = ldsa;
    a.sb = sb;
    a.c = c;
    a.ldc = ldc;
    a.M = M;
    a.N = N;
    a.K = K;
    a.offsets = nullptr;
    a.G = 1;
    a.status = d->status;
    a.sm_count = d->sm_count;
    a.splits = 1;
    a.bn = 256;   // each promotion warp then holds whole 128-column blocks of a row
    if (workspace && aligned16(workspace)) {
        a.workspace = workspace;
        a.ws_bytes = ws_bytes;
    }
    a.qout.q = qc;
    a.qout.ldq = ldqc;
    a.qout.s = sc;
    a.qout.lds = ldsc;
    a.qout.pow2 = out_mode == FP8_SCALE_POW2 ? 1 : 0;
    a.qout.write_c = c ? 1 : 0;
    if (fp8_status e = tensor_map(qa, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, lda, 128, 128,
                                  CU_TENSOR_MAP_SWIZZLE_128B, &a.tm_a))
        return e;
    if (fp8_status e = tensor_map(qb, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, N, ldb, 128, 256,
                                  CU_TENSOR_MAP_SWIZZLE_128B, &a.tm_b))
        return e;
    if (c) {
        if (fp8_status e = tensor_map(c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M, ldc * 2, 32, 32,
                                      CU_TENSOR_MAP_SWIZZLE_64B, &a.tm_c))
            return e;
    }
    if (fp8_status e = tensor_map(qc, CU_TENSOR_MAP_DATA_TYPE_UINT8, N, M, ldqc, 64, 32, CU_TENSOR_MAP_SWIZZLE_64B,
                                  &a.tm_q))
        return e;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return cuda_status(mx ? launch_gemm_mx(a, st) : launch_gemm_promote(a, st));
}

fp8_status fp8_blockscaled_grouped_gemm(const uint8_t* qa, int64_t lda, const float* sa, int64_t ldsa,
                                        const int32_t* offsets, int32_t G, int64_t M_total, const uint8_t* qb,
                                        const float* sb, void* c, int64_t ldc, int64_t N, int64_t K, uint32_t flags,
                                        void* workspace, size_t ws_bytes, fp8_stream_t stream) {
    (void)workspace;
    (void)ws_bytes;
    if (G < 1 || G > 1024) return FP8_ERR_SHAPE;
    if (fp8_status e = check_gemm_common(qa, lda, sa, ldsa, qb, sb, c, ldc, M_total, N, K, flags)) return e;
    const uint32_t path = grouped_path(flags);
    if (path == FP8_GEMM_PATH_SKINNY) return FP8_ERR_NOT_IMPLEMENTED;
    if ((flags & FP8_GEMM_SCALES_E8) && path != FP8_GEMM_PATH_MX) return FP8_ERR_NOT_IMPLEMENTED;
    if (M_total == 0) return FP8_OK;
    if (!offsets) return FP8_ERR_NULL;
    if ((int64_t)G * N > INT32_MAX) return FP8_ERR_SHAPE;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    GemmArgs a{};
    fault_injection(&a.wait_ns, &a.skip_first_load);
    a.sa = sa;
    a.ldsa = ldsa;
    a.sb = sb;
    a.c = c;
    a.ldc = ldc;
    a.M = M_total;
    a.N = N;
    a.K = K;
    a.offsets = offsets;
    a.G = G;
    a.status = d->status;
    a.sm_count = d->sm_count;
    a.splits = 1;
    const bool mx = path == FP8_GEMM_PATH_MX;
    a.scales_e8 = (flags & FP8_GEMM_SCALES_E8) ? 1 : 0;
    a.bn = mx ? kMxTileN : promote_tile_n(M_total, N, K, G);
    if (fp8_status e = tensor_map(c, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, N, M_total, ldc * 2, 32, 32,
                                  CU_TENSOR_MAP_SWIZZLE_64B, &a.tm_c))
        return e;
    if (fp8_status e = tensor_map(qa, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M_total, lda, 128, 128,
                                  CU_TENSOR_MAP_SWIZZLE_128B, &a.tm_a))
        return e;
    if (fp8_status e = tensor_map(qb, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, (uint64_t)G * N, K, 128, (uint32_t)a.bn,
                                  CU_TENSOR_MAP_SWIZZLE_128B, &a.tm_b))
        return e;
    cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
    return cuda_status(mx ? launch_gemm_mx(a, st) : launch_gemm_promote(a, st));
}

fp8_status fp8_blockscaled_gemm_skinny_noalloc(const uint8_t* qa, int64_t lda, const float* sa, int64_t ldsa,
                                               const uint8_t* qb, int64_t ldb, const float* sb, void* c,
                                               int64_t ldc, int64_t M, int64_t N, int64_t K, uint32_t flags,
                                               fp8_stream_t stream) {
    if (fp8_status e = check_gemm_common(qa, lda, sa, ldsa, qb, sb, c, ldc, M, N, K, flags)) return e;
    const uint32_t path = flags & FP8_GEMM_PATH_MASK;
    if (path != FP8_GEMM_PATH_AUTO && path != FP8_GEMM_PATH_SKINNY) return FP8_ERR_SCALE_MODE;
    if (flags & FP8_GEMM_SCALES_E8) return FP8_ERR_NOT_IMPLEMENTED;   // the skinny kernel reads fp32 scales
    if (M == 0) return FP8_OK;
    if (M > 256 || K / 128 > 1024) return FP8_ERR_SHAPE;
    if (ldb < K) return FP8_ERR_SHAPE;
    if (ldb % 16) return FP8_ERR_ALIGN;
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    GemmArgs a{};
    fault_injection(&a.wait_ns, &a.skip_first_load);
    a.sa = sa;
    a.ldsa = ldsa;
    a.sb = sb;
    a.c = c;
    a.ldc = ldc;
    a.M = M;
    a.N = N;
    a.K = K;
    a.offsets = nullptr;
    a.G = 1;
    a.status = d->status;
    a.sm_count = d->sm_count;
    a.splits = skinny_splits(M, N, K, d->sm_count);
    if (skinny_workspace_bytes(M, N, K, a.splits) > kNoAllocScratchBytes) return FP8_ERR_WORKSPACE;
    a.qb = qb;
    a.ldb = ldb;
    const int nt = skinny_tile_n(M);
    if (fp8_status e = tensor_map(qa, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, M, lda, 128, nt, CU_TENSOR_MAP_SWIZZLE_128B,
                                  &a.tm_a))
        return e;
    if (fp8_status e = tensor_map(qb, CU_TENSOR_MAP_DATA_TYPE_UINT8, K, N, ldb, 128, 128, CU_TENSOR_MAP_SWIZZLE_128B,
                                  &a.tm_b))
        return e;
    return cuda_status(launch_gemm_skinny_noalloc(a, reinterpret_cast<cudaStream_t>(stream)));
}

fp8_status fp8_debug_inject(int32_t skip_first_load, uint64_t wait_limit_ns) {
    if (wait_limit_ns > kWaitLimitNs) return FP8_ERR_SHAPE;
    g_inject_wait_ns.store(wait_limit_ns, std::memory_order_relaxed);
    g_inject_skip.store(skip_first_load ? 1 : 0, std::memory_order_relaxed);
    return FP8_OK;
}

fp8_status fp8_last_device_status(fp8_stream_t stream) {
    DeviceInfo* d;
    if (fp8_status e = current_device(&d)) return e;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) return FP8_ERR_CUDA;
    int v = 0;
    if (cudaMemcpy(&v, d->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) return FP8_ERR_CUDA;
    if (v != 0 && cudaMemset(d->status, 0, sizeof(int)) != cudaSuccess) return FP8_ERR_CUDA;
    return static_cast<fp8_status>(v);
}

}  // extern "C"
