// Definitions shared by the host dispatch (api.cu) and the kernel translation
// units: kernel argument blocks, launch entry points, device error codes.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace fa {

// Device error word codes (first error wins).  A wait time-out records
// kErrWaitTimeout | site, where `site` names the wait that gave up.
constexpr unsigned int kErrWaitTimeout = 0x1000u;

// Default limit of one bounded wait inside a kernel.  Healthy waits last
// microseconds; the limit only bounds how long a broken pipeline can stall.
constexpr unsigned long long kWaitLimitNs = 2000000000ull;

// ----------------------------------------------------------- prefill ----

struct PrefillArgs {
    float* lse;                 // [B, Hq, Sq] fp32
    const int* seqlens_k;       // [B] int32 or nullptr
    unsigned int* err_word;     // device error word
    int B, Hq, Hkv, Sq, Sk;
    int group;                  // Hq / Hkv
    int num_mblk;               // CTAs along the query axis per (b, h)
    float scale_log2;           // scale * log2(e)
    unsigned long long wait_limit_ns;
    // Debug trace (nullptr in normal use): one thread per role of CTA
    // `trace_block` (linear block index) records SM clock stamps.
    unsigned long long* trace;
    int trace_block;
};

// Trace layout: kTraceSlots stamps per role; role r, event e of iteration j
// lands at trace[r * kTraceSlots + j * kTraceEvents + e].
constexpr int kTraceSlots = 4096;
constexpr int kTraceEvents = 16;
enum TraceRole { kTrMma = 0, kTrSoftmax0 = 1, kTrSoftmax1 = 2, kTrCorr = 3, kTrLoad = 4 };

struct PrefillLaunch {
    CUtensorMap tm_q, tm_k, tm_v, tm_o;   // 3-D maps {d, S, B*H}, box {64, 128, 1}
    PrefillArgs args;
    int head_dim;
    int causal;
};

// Query rows handled by one CTA of the prefill kernel for a head dimension.
inline int prefill_rows_per_cta(int head_dim) { return head_dim <= 128 ? 256 : 128; }

cudaError_t launch_prefill_d64(const PrefillLaunch& p, cudaStream_t s);
cudaError_t launch_prefill_d96(const PrefillLaunch& p, cudaStream_t s);
cudaError_t launch_prefill_d128(const PrefillLaunch& p, cudaStream_t s);
cudaError_t launch_prefill_d256(const PrefillLaunch& p, cudaStream_t s);

// ------------------------------------------------------------ decode ----

struct DecodeArgs {
    const uint16_t* q;          // [B, Hq, Sq, d] bf16 bits
    const uint16_t* k;          // [B, Hkv, Sk, d]
    const uint16_t* v;          // [B, Hkv, Sk, d]
    uint16_t* o;                // [B, Hq, Sq, d]
    float* lse;                 // [B, Hq, Sq]
    const int* seqlens_k;       // [B] or nullptr
    float* part_o;              // [n_splits, B, Hq, Sq, d] fp32 workspace
    float* part_lse;            // [n_splits, B, Hq, Sq] fp32 workspace (log2 units)
    int B, Hq, Hkv, Sq, Sk;
    int group;                  // Hq / Hkv
    int rows;                   // group * Sq query rows per key/value head
    int n_mtiles;               // ceil(rows / 16)
    int n_splits;
    int chunk;                  // keys per split (multiple of 64)
    int causal;
    float scale_log2;
};

cudaError_t launch_decode(const DecodeArgs& a, int head_dim, cudaStream_t s);

// Fills O = 0 and LSE = -inf (used when there are no keys at all).
cudaError_t launch_fill_empty(uint16_t* o, float* lse, long long rows, int head_dim,
                              cudaStream_t s);

// Self-tests of the tcgen05 building blocks (selftest.cu).
cudaError_t launch_selftest_tmem_roundtrip(const float* in, float* out, cudaStream_t s);
cudaError_t launch_selftest_mma_tile(const uint16_t* a, const uint16_t* b, float* d, int mode,
                                     int kdim, unsigned int* err_word, cudaStream_t s);

cudaError_t launch_selftest_exp2_poly(const float* x, float* y, int n, cudaStream_t s);

// Self-test kernel for the bounded-wait path.
cudaError_t launch_wait_timeout_selftest(unsigned int* err_word, unsigned long long limit_ns,
                                         cudaStream_t s);

}  // namespace fa
