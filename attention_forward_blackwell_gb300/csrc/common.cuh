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
    uint16_t* o;                // [B, Hq, Sq, d] bf16 bits (written directly by merges)
    float* lse;                 // [B, Hq, Sq] fp32
    const int* seqlens_k;       // [B] int32 or nullptr
    unsigned int* err_word;     // device error word
    int B, Hq, Hkv, Sq, Sk;
    int group;                  // Hq / Hkv
    int window;                 // sliding window in keys (<= 0: none)
    const float* sinks;         // [Hq] sink logits (scaled-score units) or nullptr
    // Paged K/V (nullptr: contiguous [B, Hkv, Sk, d]): the caches are
    // [num_pages, Hkv, page_size, d] and key j of sequence b is row
    // j % page_size of page block_table[b * max_pages + j / page_size];
    // page_size is a multiple of the 128-key tile, so a tile never crosses a
    // page.
    const int* block_table;
    int max_pages;
    int page_size;
    // Packed variable-length sequences (nullptr: dense): sequence b owns
    // query tokens [cu_seqlens_q[b], cu_seqlens_q[b+1]) of Q, O [total_q, Hq, d]
    // and keys [cu_seqlens_k[b], cu_seqlens_k[b+1]) of K, V [total_k, Hkv, d]
    // (with paged caches instead: seqlens_k[b] keys through the block table);
    // LSE is [Hq, total_q].  Offsets are clamped to [0, total] in the kernel.
    // Sq is then the largest query length (units per (b, h) = num_mblk).
    const int* cu_seqlens_q;
    const int* cu_seqlens_k;
    int total_q, total_k;
    int num_mblk;               // query blocks (units) per (b, h)
    // Query heads per tile of the 256-key kernel (1: one head per unit).
    // With pack = P > 1 a unit's 128 tile rows are P consecutive query heads
    // of one kv group x 128 / P query positions (row r: head h + r / (128 / P),
    // position row0 + r % (128 / P)), and num_mblk counts units per (b, group
    // of P heads).
    int pack;
    // Work split (see prefill_work): CTAs [0, n_full) process whole units;
    // each later unit is split into `split` pieces of its nk key blocks.
    int n_full;
    int split;
    int n_work;                 // work items of a persistent launch: n_full + n_tail * split
    int nk;                     // key blocks of a unit, ceil(Sk / keys per block)
    // Scratch of the split units (nullptr when nothing is split): partial O
    // of every piece, [pieces][NQ][d / 4][128][4] fp32, its row max and row
    // sum, [pieces][NQ][2][128] fp32, and one arrival counter per split unit,
    // tagged with `epoch` (a value no earlier launch used) so that stale
    // counter contents never count.
    float* part_o;
    float* part_ml;
    unsigned long long* part_count;
    unsigned long long epoch;
    float scale_log2;           // scale * log2(e)
    // The producer of CTA c prefetches into L2 the Q tiles of CTA
    // c + q_prefetch (dispatched about one wave later), 0: none.
    int q_prefetch;
    unsigned long long wait_limit_ns;
    // Debug trace (nullptr in normal use): one thread per role of CTA
    // `trace_block` (linear block index) records SM clock stamps.
    unsigned long long* trace;
    int trace_block;
};

#ifndef FA_PREFILL_TRACE
#define FA_PREFILL_TRACE 0   // 1: compile the prefill kernel's clock trace
#endif
// Trace layout: kTraceSlots stamps per role; role r, event e of iteration j
// lands at trace[r * kTraceSlots + j * kTraceEvents + e].
constexpr int kTraceSlots = 4096;
constexpr int kTraceEvents = 16;
enum TraceRole { kTrMma = 0, kTrSoftmax0 = 1, kTrSoftmax1 = 2, kTrCorr = 3, kTrLoad = 4 };

struct PrefillLaunch {
    CUtensorMap tm_q, tm_k, tm_v, tm_o;   // 3-D maps {d, S, B*H}, box {64, 128, 1}
    CUtensorMap tm_o32;                   // persistent kernels: O, box {32, 32, 1}, 64-byte swizzle
    PrefillArgs args;
    int n_tail;                 // split units
    int head_dim;
    int causal;
    int num_sms;                // SMs of the device (CTAs of a persistent launch)
    int wide;                   // prefill_wide_ok: 256-key score blocks (units of 128 query
                                // rows, tm_k box {64, 256, 1}, tm_o32 set)
};

// The 256-key persistent kernel (head_dim 96 and 128) takes dense launches,
// causal or not: no window, contiguous K/V (no block table), no packed
// sequences.
inline bool prefill_wide_ok(int head_dim, int window, bool paged, bool packed) {
    return (head_dim == 96 || head_dim == 128) && window <= 0 && !paged && !packed;
}
// Query heads that share one 128-row tile of the 256-key kernel (GQA head
// packing): rows per head R = the next power of two >= sq, at least 16, and
// P = 128 / R heads of the group (P a power of two dividing it); short query
// lengths then fill the tile with the group's other heads, which read the
// same keys, instead of leaving most of its rows empty.
inline int prefill_pack(int sq, int group) {
    int rows = 16;
    while (rows < sq && rows < 128) rows *= 2;
    int p = 128 / rows;
    while (p > 1 && (group % p) != 0) p /= 2;
    return p;
}
// Query rows of one prefill unit (query block) for a head dimension.
inline int prefill_rows_per_cta(int head_dim) { return head_dim <= 128 ? 256 : 128; }
// CTAs per unit: head_dim 512 shares the output columns out over two.
inline int prefill_ctas_per_unit(int head_dim) { return head_dim == 512 ? 2 : 1; }
// Head dimensions of the prefill kernels.
inline bool prefill_head_dim_ok(int head_dim) {
    return head_dim == 64 || head_dim == 96 || head_dim == 128 || head_dim == 256 ||
           head_dim == 512;
}

// Split of the prefill work over the grid.  With units of equal work
// (non-causal), the units beyond the last full wave of `ctas` whole-unit
// CTAs (all units if there are fewer than `ctas`) are cut into `split`
// pieces along the key axis: the largest split whose pieces all run in one
// wave (tail * split <= ctas) with at least 8 key blocks per piece and at
// most 8 pieces, so that the last wave is `split` times shorter (measured on
// GB300: more pieces than one wave holds, or shorter pieces, lose more to
// per-CTA set-up and to the merge than they gain).  Causal units start
// heaviest first and are not split.
struct PrefillPlan {
    int n_full;   // CTAs that process a whole unit
    int n_tail;   // units processed in pieces
    int split;    // pieces per such unit (1: nothing is split)
};

inline PrefillPlan plan_prefill(long long units, int nk, int causal, int ctas) {
    PrefillPlan p{(int)units, 0, 1};
    if (causal || units <= 0 || ctas <= 0) return p;
    const long long tail = units % ctas;
    if (tail == 0) return p;
    long long k = ctas / tail;
    if (k > nk / 8) k = nk / 8;
    if (k > 8) k = 8;
    if (k < 2) return p;
    p.n_full = (int)(units - tail);
    p.n_tail = (int)tail;
    p.split = (int)k;
    return p;
}

// How a prefill launch is cut into work: which kernel family runs it, the
// query rows of a unit, the keys of a score block and the work split.  One
// function serves the launch and the plan queries, so that they agree.
struct PrefillShape {
    bool wide;             // prefill_wide_ok: the 256-key persistent kernel
    int pack;              // query heads per unit (prefill_pack; 1 unless wide)
    int rows_per_unit;     // query rows of a unit (query block), per head
    int keys_per_block;    // keys of a score block
    int num_mblk;          // units per (batch entry, query head)
    long long units;
    int nk;                // key blocks of a unit
    PrefillPlan plan;
    bool persistent;       // one CTA per SM walks the unit list
};

// group: query heads per kv head (1: no head packing).
inline PrefillShape prefill_shape(int batch, int hq, int sq, int sk, int head_dim, bool causal,
                                  int window, bool paged, bool packed, int num_sms,
                                  int group = 1) {
    PrefillShape s;
    s.wide = prefill_wide_ok(head_dim, window, paged, packed);
    s.pack = s.wide ? prefill_pack(sq, group > 0 ? group : 1) : 1;
    s.rows_per_unit = s.wide ? 128 / s.pack : prefill_rows_per_cta(head_dim);
    s.keys_per_block = s.wide ? 256 : 128;
    s.num_mblk = (sq + s.rows_per_unit - 1) / s.rows_per_unit;
    s.units = (long long)batch * (hq / s.pack) * s.num_mblk;
    s.nk = (sk + s.keys_per_block - 1) / s.keys_per_block;
    // not split: causal units (heaviest first), windowed ones (fewer key
    // blocks than nk), packed sequences (units of different lengths), head_dim
    // 512 (two CTAs per unit already)
    s.plan = plan_prefill(s.units, s.nk,
                          causal || window > 0 || packed || head_dim == 512 || s.wide, num_sms);
    // the 256-key kernel with at most half a wave of (non-causal) units: each
    // unit in `split` pieces of >= 4 key blocks, one piece per CTA, so that
    // the SMs the units leave idle share the keys (the last piece to finish
    // merges); with more units it walks them whole
    if (s.wide && !causal && s.units > 0 && s.units * 2 <= num_sms) {
        long long k = num_sms / s.units;
        if (k > 8) k = 8;
        if (k > s.nk / 4) k = s.nk / 4;
        if (k >= 2) s.plan = PrefillPlan{0, (int)s.units, (int)k};
    }
    // head_dim 256 launches of whole units, and the 256-key kernel, run one
    // persistent CTA per SM
    s.persistent = s.wide || (head_dim == 256 && !packed && s.plan.n_tail == 0 &&
                              s.plan.n_full > 0 && num_sms > 0);
    return s;
}

cudaError_t launch_prefill_d64(const PrefillLaunch& p, cudaStream_t s);
cudaError_t launch_prefill_d96(const PrefillLaunch& p, cudaStream_t s);
cudaError_t launch_prefill_d128(const PrefillLaunch& p, cudaStream_t s);
cudaError_t launch_prefill_d256(const PrefillLaunch& p, cudaStream_t s);
cudaError_t launch_prefill_d512(const PrefillLaunch& p, cudaStream_t s);

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
    int window;                 // sliding window in keys (<= 0: none)
    const float* sinks;         // [Hq] sink logits (scaled-score units) or nullptr
    // Paged K/V (nullptr: contiguous): caches [num_pages, Hkv, page_size, d],
    // key j of sequence b at row j % page_size of page
    // block_table[b * max_pages + j / page_size] (clamped to the cache).
    const int* block_table;
    int max_pages;
    int page_size;
    int num_pages;
    float scale_log2;
};

cudaError_t launch_decode(const DecodeArgs& a, int head_dim, cudaStream_t s);

// Fills O = 0 and LSE = -inf, or the row's sink logit when sinks is not null
// (used when there are no keys at all); rows are ordered (b, h < hq, i < sq).
cudaError_t launch_fill_empty(uint16_t* o, float* lse, long long rows, int head_dim,
                              const float* sinks, int hq, int sq, cudaStream_t s);

// Self-tests of the tcgen05 building blocks (selftest.cu).
cudaError_t launch_selftest_tmem_roundtrip(const float* in, float* out, cudaStream_t s);
cudaError_t launch_selftest_mma_tile(const uint16_t* a, const uint16_t* b, float* d, int mode,
                                     int kdim, unsigned int* err_word, cudaStream_t s);

cudaError_t launch_selftest_exp2_poly(const float* x, float* y, int n, cudaStream_t s);

// Self-test kernel for the bounded-wait path.
cudaError_t launch_wait_timeout_selftest(unsigned int* err_word, unsigned long long limit_ns,
                                         cudaStream_t s);

}  // namespace fa
