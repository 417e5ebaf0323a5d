// Host-side interface between the C-ABI layer (api.cu) and the kernel
// translation units.  Not part of the public ABI.
#pragma once
#include <atomic>
#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fp8bs {

// Every GEMM workspace starts with this many bytes of split-K / last-wave
// tickets (int32, zero between calls: each call leaves the ones it used at
// zero); the fp32 partials of every path start after it, so one call's
// partials never land on the tickets another call relies on.
constexpr size_t kTicketBytes = size_t(64) << 10;
constexpr int64_t kMaxTickets = (int64_t)(kTicketBytes / sizeof(int32_t));

// Upper bound on any single wait inside a kernel before it records a timeout
// and returns (nanoseconds of %globaltimer).
constexpr uint64_t kWaitLimitNs = 2000000000ull;   // 2 s

// Launches `kern` with programmatic stream serialization: it may start while
// the previous kernel in the stream finishes, and waits for it in
// griddep_wait() (the kernel must call that before touching its inputs).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                       Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<Args&&>(args)...);
}

// Decode-sized steps (activation quantiser + skinny GEMM) launch with
// programmatic stream serialization: measured 7-12% faster per layer at
// 1..8 tokens, but 1.5-6% slower at 64..256 tokens with K = 14336.
inline bool pdl_for_tokens(int64_t M) { return M <= 32; }

// Per-device "done once" flags for a kernel's attribute set-up, safe to query
// from several host threads (devices past 63 redo the set-up on every call,
// which is harmless).
struct DeviceOnce {
    std::atomic<bool> done[64];
    bool test(int dev) const { return dev >= 0 && dev < 64 && done[dev].load(std::memory_order_acquire); }
    void set(int dev) {
        if (dev >= 0 && dev < 64) done[dev].store(true, std::memory_order_release);
    }
};

// Codes written to the per-device status word (same values as fp8_status).
constexpr int kStatusTimeout = 8;

struct DeviceInfo {
    int device = -1;
    int sm_count = 0;
    int max_smem_optin = 0;
    int* status = nullptr;          // device address of the status word
};

// ------------------------------------------------------------- quantisers
// s8 != nullptr: power-of-two scales written as UE8M0 bytes there (s unused).
cudaError_t launch_quant_act_1x128(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq,
                                   float* s, int64_t lds, bool pow2, cudaStream_t st, uint8_t* s8 = nullptr);
cudaError_t launch_quant_act_weight(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* qa, int64_t ldqa,
                                    float* sa, int64_t ldsa, const void* w, int64_t N, int64_t ldw, uint8_t* qw,
                                    int64_t ldqw, float* sw, bool pow2, cudaStream_t st);
cudaError_t launch_quant_weight_128x128(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q,
                                        int64_t ldq, float* s, bool pow2, cudaStream_t st, uint8_t* s8 = nullptr);

// Transposing quantisers (training-side GEMM operands).  q == nullptr: the
// non-transposed codes and scales are not written.
cudaError_t launch_quant_act_128x1(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* qt, int64_t ldqt,
                                   float* st, int64_t ldst, uint8_t* q, int64_t ldq, float* s, int64_t lds,
                                   bool pow2, cudaStream_t stream);
// Grouped 128x1 quantiser (mixture-of-experts weight gradients): each
// expert's tokens in 128x1 blocks of their own, written to padded token slots
// (see quant_t.cu).  grouped_token_blocks(T, G): the padded blocks an
// expert-sorted T-token batch can need at most (the grid, and the columns of
// qt / 128 and rows of st the caller provides).
constexpr int kMaxGroupedQuantExperts = 1024;
inline int64_t grouped_token_blocks(int64_t T, int64_t G) { return (T + 127) / 128 + G; }
cudaError_t launch_quant_act_128x1_grouped(const void* x, int64_t T, int64_t K, int64_t ldx, const int32_t* offsets,
                                           int32_t G, uint8_t* qt, int64_t ldqt, float* st, int64_t ldst, bool pow2,
                                           cudaStream_t stream);
cudaError_t launch_quant_weight_128x128_t(const void* w, int64_t N, int64_t K, int64_t ldw, uint8_t* q, int64_t ldq,
                                          float* s, uint8_t* qt, int64_t ldqt, float* st, bool pow2,
                                          cudaStream_t stream);

// Per-tensor quantiser: zeroes scale_amax[1], reduces max |x| into it, then
// casts with the scale it derives (written to scale_amax[0]).
cudaError_t launch_quant_per_tensor(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq,
                                    float* scale_amax, bool pow2, int sm_count, cudaStream_t st);

cudaError_t launch_cast_with_scale(const void* x, int64_t M, int64_t K, int64_t ldx, uint8_t* q, int64_t ldq,
                                   const float* scale, int sm_count, cudaStream_t st);

// FP8 KV cache decode attention (attn.cu): D = 128, Hq / Hkv in {1, 2, 4, 8}.
int attn_splits(int T);
cudaError_t launch_kv_append(const void* k_new, const void* v_new, const float* sk, const float* sv,
                             const int32_t* seq_lens, uint8_t* kc, uint8_t* vc, int B, int Hkv, int T,
                             cudaStream_t st);
size_t attn_workspace_bytes(int B, int Hq, int T);
cudaError_t launch_decode_attention(const uint8_t* q, const float* sq, const uint8_t* kc, const float* sk,
                                    const uint8_t* vc, const float* sv, const int32_t* seq_lens, int B, int Hq,
                                    int Hkv, int T, void* workspace, uint16_t* out, cudaStream_t st);

// ------------------------------------------------------------- GEMMs
// Fused quantisation of the GEMM's output for the next layer: the E4M3 codes
// and 1x128 scales fp8_quant_act_1x128 would produce from the bf16 C.
struct QuantOut {
    uint8_t* q;         // codes [M][ldq]; nullptr: no fused quantisation
    int64_t ldq;
    float* s;           // scales, K-block-major: s[(column / 128) * lds + row]
    int64_t lds;
    int pow2;           // scale rule of the codes (FP8_SCALE_POW2)
    int write_c;        // also write the bf16 C
};

struct GemmArgs {
    CUtensorMap tm_a;               // qa [rows, K] uint8, box {128, 128}, 128B swizzle
    CUtensorMap tm_b;               // qb [rows, K] uint8, box {128, BN}, 128B swizzle
    CUtensorMap tm_c;               // promote / MX: c [rows, N] bf16, box {32, 32}, 64B swizzle
    CUtensorMap tm_q;               // promote with QuantOut: codes [rows, N] u8, box {64, 32}, 64B swizzle
    QuantOut qout;                  // promote: fused output quantisation (qout.q == nullptr: none)
    const float* sa;
    int64_t ldsa;
    const float* sb;
    int per_tensor;                 // MX only: sa, sb point at one scale each (per-tensor scaling)
    int scales_e8;                  // MX only: sa, sb hold UE8M0 bytes (same indices as the fp32 arrays)
    int64_t ldsb;                   // 0: sb holds 128x128 block scales [G][N/128][K/128];
                                    // > 0: a scale per B row, sb[kb * ldsb + n] (dense promote / MX)
    void* c;
    int64_t ldc;
    const uint8_t* qb;              // skinny: the weight codes, streamed with cp.async
    int64_t ldb;
    int64_t M, N, K;
    const int32_t* offsets;         // grouped: [G+1] on device; nullptr for dense
    int32_t G;
    int32_t kgroup;                 // promote wgrad: G GEMMs over the experts' padded token blocks
    int64_t kg_tokens;              //   (tokens the offsets range over)
    void* workspace;
    size_t ws_bytes;
    int32_t splits;
    int32_t bn;                     // promote kernel tile width (128 or 256)
    int* status;
    int sm_count;
    // failure-path test hook (fp8_debug_inject): 0 = the default wait bound
    // (kWaitLimitNs); skip_first_load != 0 makes the TMA producer skip the
    // first K-block's operands, so the waits on them run out
    uint64_t wait_ns;
    int32_t skip_first_load;
};

// The current fault-injection setting (fp8_debug_inject), copied into every
// GEMM's arguments.
void fault_injection(uint64_t* wait_ns, int32_t* skip_first_load);
inline uint64_t wait_bound(const GemmArgs& a) { return a.wait_ns ? a.wait_ns : kWaitLimitNs; }

// Dense / grouped kernel with per-K-block fp32 promotion (tcgen05, TMEM);
// output tile 128 x bn with bn = 128 or 256 (promote_tile_n picks it).
int promote_tile_n(int64_t M, int64_t N, int64_t K, int32_t G);
cudaError_t launch_gemm_promote(const GemmArgs& a, cudaStream_t st);

// Dense promote and MX kernels: the last, partial wave of tiles is split along
// K when the caller's workspace holds `bytes` (tickets first, then fp32 parts).
struct TailPlan {
    int64_t n_full;       // tiles computed whole
    int parts;            // parts per remaining tile (1: no split)
    size_t ticket_bytes;  // zero-initialised tickets at the start of the workspace
    size_t bytes;         // workspace needed for the split (0 when none)
};
constexpr int kPromoteMaxParts = 4, kMxMaxParts = 2;
constexpr int kSingleWaveMaxParts = 16;    // fewer tiles than SMs: parts per tile at most
constexpr int64_t kSkinnyAutoMaxM = 128;   // FP8_GEMM_PATH_AUTO: the skinny kernel up to this many rows
constexpr int kMxTileN = 256;   // MX kernel output tile width
TailPlan tail_plan(int64_t M, int64_t N, int64_t K, int sm_count, int bn, int max_parts);
size_t promote_workspace_bytes(int64_t M, int64_t N, int64_t K, int sm_count);

// Dense / grouped kernel for power-of-two scales: the tensor core applies the
// scales as UE8M0 block scale factors (tcgen05.mma kind::mxf8f6f4); output
// tile 128 x 256 (kMxTileN), a.tm_b with box {128, 256}, a.tm_c as noted above.  Every scale must be a power of
// two in [2^-127, 2^127]; others are reported in the status word.
cudaError_t launch_gemm_mx(const GemmArgs& a, cudaStream_t st);

// Skinny (decode) kernel: weights on the MMA's M side, tokens on N, split-K.
int skinny_tile_n(int64_t M);                         // padded token count, 0 if M > 256
int skinny_splits(int64_t M, int64_t N, int64_t K, int sm_count);
size_t skinny_workspace_bytes(int64_t M, int64_t N, int64_t K, int splits);
cudaError_t launch_gemm_skinny(const GemmArgs& a, cudaStream_t st);

// Size of the library-owned scratch of the no-allocation skinny entry point.
constexpr size_t kNoAllocScratchBytes = size_t(8) << 20;   // 8 MiB per device
// Same launch as launch_gemm_skinny with a.workspace replaced by that scratch
// (set up on the first call per device, ticket words cleared every call).
cudaError_t launch_gemm_skinny_noalloc(GemmArgs a, cudaStream_t st);

}  // namespace fp8bs
