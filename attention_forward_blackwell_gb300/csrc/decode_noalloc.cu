// Decode forward for callers that cannot allocate device memory.
//
// fa_fwd_decode takes its split partials from a stream-ordered workspace
// (cudaMallocAsync / cudaFreeAsync on every call).  Some callers cannot do
// that: a serving loop that must not allocate once it is running (an
// allocation can stall or fail at an unpredictable moment), a process whose
// device memory is already reserved by another allocator so that any fresh
// allocation would fail, or a deployment whose components must declare all
// device memory up front.  fa_fwd_decode_noalloc runs the same split and
// combine kernels, but keeps the partials in one fixed device array declared
// below, so the call itself allocates nothing.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "../../include/fa.h"
#include "common.cuh"

namespace fa {
namespace {

// Capacity of the scratch array: FA_DECODE_NOALLOC_SCRATCH_BYTES (16 MiB) of
// fp32 partials.  A call needs n_splits * batch * hq * sq * (head_dim + 1)
// floats.
constexpr size_t kNoAllocScratchFloats = FA_DECODE_NOALLOC_SCRATCH_BYTES / sizeof(float);

// Every GPU on which this library is loaded reserves this array until the
// process exits.  In host code its name is only a stand-in for the device
// symbol: the device address is obtained with cudaGetSymbolAddress below.
static __device__ __align__(256) float g_noalloc_scratch[kNoAllocScratchFloats];

struct ScratchSlot {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    float* ptr = nullptr;   // device address of g_noalloc_scratch on this device
};

constexpr int kMaxDevices = 64;
std::mutex g_mu;
ScratchSlot g_slots[kMaxDevices];

// One-time set-up per device, with that device current: query the device and
// resolve the scratch array's device address.
const ScratchSlot* scratch_slot() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    ScratchSlot& s = g_slots[dev];
    if (!s.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        s.supported = (major == 10 && minor == 3);
        s.num_sms = sms;
        if (s.supported) {
            float* p = nullptr;
            if (cudaGetSymbolAddress((void**)&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
                return nullptr;
            s.ptr = p;
        }
        s.ready = true;
    }
    return &s;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" fa_status fa_fwd_decode_noalloc(const void* q, const void* k, const void* v, void* o,
                                           float* lse, int batch, int hq, int hkv, int sq, int sk,
                                           const int* seqlens_k, int head_dim, float scale,
                                           int causal, fa_stream_t stream) {
    // argument checks: the same rules as fa_fwd_decode
    if (batch < 0 || hq < 0 || hkv < 0 || sq < 0 || sk < 0) return FA_ERR_INVALID_ARG;
    if (batch > 65535 || hq > 65535) return FA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (batch == 0 || hq == 0 || sq == 0) return FA_OK;
    if (hkv == 0 || hq % hkv != 0) return FA_ERR_INVALID_ARG;
    if (!q || !o || !lse) return FA_ERR_INVALID_ARG;
    if (sk > 0 && (!k || !v)) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(o) || (sk > 0 && (!aligned16(k) || !aligned16(v))))
        return FA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_MISALIGNED;
    if (sq > FA_DECODE_MAX_SQ) return FA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return FA_ERR_UNSUPPORTED;
    if ((long long)batch * hq * sq * head_dim >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    // the scratch must hold at least one split's partials
    const size_t rows = (size_t)batch * hq * sq;
    const size_t per_split = rows * (size_t)(head_dim + 1);
    if (sk > 0 && per_split > kNoAllocScratchFloats) return FA_ERR_INVALID_ARG;

    const ScratchSlot* slot = scratch_slot();
    if (!slot) return FA_ERR_CUDA;
    if (!slot->supported) return FA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (sk == 0)
        return launch_fill_empty(static_cast<uint16_t*>(o), lse, (long long)rows, head_dim,
                                 nullptr, hq, sq, s) ==
                       cudaSuccess
                   ? FA_OK
                   : FA_ERR_CUDA;

    DecodeArgs a{};
    a.q = static_cast<const uint16_t*>(q);
    a.k = static_cast<const uint16_t*>(k);
    a.v = static_cast<const uint16_t*>(v);
    a.o = static_cast<uint16_t*>(o);
    a.lse = lse;
    a.seqlens_k = seqlens_k;
    a.B = batch;
    a.Hq = hq;
    a.Hkv = hkv;
    a.Sq = sq;
    a.Sk = sk;
    a.group = hq / hkv;
    a.rows = a.group * sq;
    a.n_mtiles = (a.rows + 15) / 16;
    a.causal = causal ? 1 : 0;
    a.scale_log2 = scale * 1.4426950408889634f;
    if ((long long)hkv * a.n_mtiles > 65535) return FA_ERR_INVALID_ARG;
    // split plan: as many splits as keep the GPU busy, but no more than fit
    // the scratch array
    const long long pairs = (long long)batch * hkv * a.n_mtiles;
    long long want = (24ll * slot->num_sms + pairs - 1) / pairs;
    const long long max_by_keys = (sk + 255) / 256;
    const long long max_by_scratch = (long long)(kNoAllocScratchFloats / per_split);
    if (want > max_by_keys) want = max_by_keys;
    if (want > max_by_scratch) want = max_by_scratch;
    if (want < 1) want = 1;
    long long chunk = ((long long)sk + want - 1) / want;
    chunk = (chunk + 63) / 64 * 64;
    a.chunk = (int)chunk;
    a.n_splits = (int)((sk + chunk - 1) / chunk);
    // every partial the combine kernel reads is written by the split kernel
    // of the same call, so the array needs no clearing between calls
    a.part_o = slot->ptr;
    a.part_lse = slot->ptr + (size_t)a.n_splits * rows * head_dim;
    return launch_decode(a, head_dim, s) == cudaSuccess ? FA_OK : FA_ERR_CUDA;
}
