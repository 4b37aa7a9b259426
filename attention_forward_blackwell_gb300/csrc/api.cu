// C ABI of libfa_gb300.so (declared in include/fa.h): argument validation,
// device checks, TMA tensor-map encoding, split planning and kernel dispatch.
// Everything runs on the host and only enqueues work on the caller's stream.
#include <cmath>
#include <cstdint>
#include <cstdio>
#include <cstdlib>
#include <algorithm>
#include <atomic>
#include <mutex>

#include "../../include/fa.h"
#include "common.cuh"

namespace fa {
namespace {

// Device error word written by kernels whose bounded waits give up.
__device__ unsigned int g_err_word;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
    bool ready = false;
    bool supported = false;
    int num_sms = 0;
    unsigned int* err_word = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                  const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                  const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;

// Debug trace target of the next prefill launches (see fa_debug_prefill_trace).
unsigned long long* g_trace_buf = nullptr;
int g_trace_block = 0;

// Looks up (once) the properties of the current device.  Returns nullptr if
// the CUDA runtime fails.
const DeviceInfo* device_info() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return nullptr;
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceInfo& di = g_dev[dev];
    if (!di.ready) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
            return nullptr;
        di.supported = (major == 10 && minor == 3);
        di.num_sms = sms;
        if (di.supported) {
            void* p = nullptr;
            if (cudaGetSymbolAddress(&p, g_err_word) != cudaSuccess) return nullptr;
            di.err_word = static_cast<unsigned int*>(p);
            // keep stream-ordered workspace blocks cached between calls
            cudaMemPool_t pool;
            if (cudaDeviceGetDefaultMemPool(&pool, dev) == cudaSuccess) {
                uint64_t thr = UINT64_MAX;
                cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &thr);
            }
        }
        if (!g_encode) {
            void* fn = nullptr;
            cudaDriverEntryPointQueryResult q;
            if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000,
                                                 cudaEnableDefault, &q) != cudaSuccess ||
                q != cudaDriverEntryPointSuccess || fn == nullptr)
                return nullptr;
            g_encode = reinterpret_cast<EncodeTiledFn>(fn);
        }
        di.ready = true;
    }
    return &di;
}

// Tags of the split-unit arrival counters: a 48-bit value no earlier launch
// of this process used, so counters left in reused scratch never match.
unsigned long long next_prefill_epoch() {
    static std::atomic<unsigned long long> counter{0};
    const unsigned long long e = (counter.fetch_add(1) + 1) & ((1ull << 48) - 1);
    return e == 0 ? 1 : e;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// 3-D bf16 map {d, rows, planes} with a {64, box_rows, box_planes} box (128
// rows of one plane; 256 rows for the K blocks of the 256-key kernels; 128 /
// P rows of P planes for a head-packed Q tile) and 128-byte swizzle (rows
// past `rows` and columns past `d` read as zero).
// Strides in bytes: row_stride between rows, plane_stride between planes
// (contiguous [planes][rows][d] when they are d * 2 and rows * d * 2).
bool encode_map_strided(CUtensorMap* m, const void* base, int d, long long rows, long long planes,
                        unsigned long long row_stride, unsigned long long plane_stride,
                        unsigned box_rows = 128, unsigned box_planes = 1) {
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)planes};
    const cuuint64_t strides[2] = {(cuuint64_t)row_stride, (cuuint64_t)plane_stride};
    const cuuint32_t box[3] = {64, box_rows, box_planes};
    const cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 3-D bf16 map {d, rows, planes} with a {32, box_rows, 32 / box_rows} box
// (32 rows in all) and 64-byte swizzle (16-byte chunks of each 64-byte row
// XOR-ed with bits 1-2 of the row): the persistent kernels' O stores from
// 2 KB per-warp staging areas; 16 rows x 2 planes for a head-packed tile of
// 16 rows per head.
bool encode_map32_strided(CUtensorMap* m, const void* base, int d, long long rows,
                          long long planes, unsigned long long row_stride,
                          unsigned long long plane_stride, unsigned box_rows = 32) {
    const cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)rows, (cuuint64_t)planes};
    const cuuint64_t strides[2] = {(cuuint64_t)row_stride, (cuuint64_t)plane_stride};
    const cuuint32_t box[3] = {32, box_rows, 32 / box_rows};
    const cuuint32_t estr[3] = {1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_64B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// 4-D bf16 map {64 columns, rows, d / 64 chunks, planes} (chunk stride 128
// bytes) with a {64, 128, 2, 1} box: one copy brings two 64-column chunks of
// a 128-row tile, written to shared memory as [chunk][row][64 columns] with
// 128-byte swizzle, the same bytes as two boxes of the 3-D map.  d must be a
// multiple of 128.
bool encode_map4_strided(CUtensorMap* m, const void* base, int d, long long rows, long long planes,
                         unsigned long long row_stride, unsigned long long plane_stride,
                         unsigned box_rows = 128, unsigned box_chunks = 2) {
    const cuuint64_t dims[4] = {64, (cuuint64_t)rows, (cuuint64_t)(d / 64), (cuuint64_t)planes};
    const cuuint64_t strides[3] = {(cuuint64_t)row_stride, 128, (cuuint64_t)plane_stride};
    const cuuint32_t box[4] = {64, box_rows, box_chunks, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(base), dims, strides,
                    box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Load maps of the prefill kernels: 4-D (two chunks per copy) for head_dim
// 256, 3-D otherwise.  The V maps of head_dim 256 and 512 copy 64 / 32 rows
// x four 64-column chunks at a time (the kernels' row-split value slots).
bool prefill_load_map(CUtensorMap* m, const void* base, int d, long long rows, long long planes,
                      unsigned long long row_stride, unsigned long long plane_stride,
                      bool value = false) {
    if (d == 256)
        return value ? encode_map4_strided(m, base, d, rows, planes, row_stride, plane_stride, 64, 4)
                     : encode_map4_strided(m, base, d, rows, planes, row_stride, plane_stride);
    if (d == 512 && value)
        return encode_map4_strided(m, base, d, rows, planes, row_stride, plane_stride, 32, 4);
    return encode_map_strided(m, base, d, rows, planes, row_stride, plane_stride);
}

bool encode_map(CUtensorMap* m, const void* base, int d, int rows, long long planes) {
    return encode_map_strided(m, base, d, rows, planes, (unsigned long long)d * 2,
                              (unsigned long long)rows * d * 2);
}

struct Common {
    bool noop = false;   // nothing to compute
};

// Checks shared by prefill and decode; fills `c.noop`.
fa_status check_common(const void* q, const void* k, const void* v, void* o, float* lse,
                       int batch, int hq, int hkv, int sq, int sk, float scale, Common& c) {
    if (batch < 0 || hq < 0 || hkv < 0 || sq < 0 || sk < 0) return FA_ERR_INVALID_ARG;
    if (batch > 65535 || hq > 65535) return FA_ERR_INVALID_ARG;
    if (!(scale > 0.f) || !std::isfinite(scale)) return FA_ERR_INVALID_ARG;
    if (batch == 0 || hq == 0 || sq == 0) {
        c.noop = true;
        return FA_OK;
    }
    if (hkv == 0 || hq % hkv != 0) return FA_ERR_INVALID_ARG;
    if (!q || !o || !lse) return FA_ERR_INVALID_ARG;
    if (sk > 0 && (!k || !v)) return FA_ERR_INVALID_ARG;
    if (!aligned16(q) || !aligned16(o) || (sk > 0 && (!aligned16(k) || !aligned16(v))))
        return FA_ERR_MISALIGNED;
    if ((reinterpret_cast<uintptr_t>(lse) & 3u) != 0) return FA_ERR_MISALIGNED;
    return FA_OK;
}

fa_status from_cuda(cudaError_t e) { return e == cudaSuccess ? FA_OK : FA_ERR_CUDA; }

// Checks of the paged-cache arguments shared by prefill and decode.
fa_status check_paged(const int* seqlens_k, const int* block_table, int max_pages, int page_size,
                      int num_pages, int batch, int hq, int sq) {
    if (batch == 0 || hq == 0 || sq == 0) return FA_OK;   // nothing to compute
    if (!seqlens_k || !block_table) return FA_ERR_INVALID_ARG;
    if (max_pages <= 0 || page_size <= 0 || num_pages <= 0) return FA_ERR_INVALID_ARG;
    if ((long long)max_pages * page_size >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(block_table) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(seqlens_k) & 3u) != 0)
        return FA_ERR_MISALIGNED;
    return FA_OK;
}

struct Varlen;
fa_status prefill_impl(const void* q, const void* k, const void* v, void* o, float* lse, int batch,
                       int hq, int hkv, int sq, int sk, const int* seqlens_k, int head_dim,
                       float scale, int causal, int window, const float* sinks,
                       const int* block_table, int max_pages, int page_size, int num_pages,
                       fa_stream_t stream, const Varlen* vl);

// Query rows per kv head (G * sq) from which a decode call at head_dim 128
// runs the head-packed prefill kernel instead of the split-KV kernel.  Past
// 16 rows per kv head the split kernel's query tiles (16 rows each on
// mma.sync) make it compute-bound (B=64, Hq=64, Hkv=8, key lengths 1K-16K:
// 6497 / 6353 / 5169 / 3086 / 1707 GB/s at sq = 1 / 2 / 4 / 8 / 16, the
// packed kernel 5169-5244 throughout); with few units the packed kernel
// splits them along the keys over the idle SMs, so that at 16K keys it is
// 1.2-3.9x faster for every batch from 1 to 16 at 32 to 128 rows.
constexpr int kDecodeToPrefillRows = 32;

fa_status decode_impl(const void* q, const void* k, const void* v, void* o, float* lse, int batch,
                      int hq, int hkv, int sq, int sk, const int* seqlens_k, int head_dim,
                      float scale, int causal, int window, const float* sinks, int num_splits,
                      fa_stream_t stream, const int* block_table = nullptr, int max_pages = 0,
                      int page_size = 0, int num_pages = 0) {
    Common c;
    fa_status st = check_common(q, k, v, o, lse, batch, hq, hkv, sq, sk, scale, c);
    if (st != FA_OK || c.noop) return st;
    if ((reinterpret_cast<uintptr_t>(sinks) & 3u) != 0) return FA_ERR_MISALIGNED;
    if (sq > FA_DECODE_MAX_SQ) return FA_ERR_INVALID_ARG;
    if (head_dim != 64 && head_dim != 128 && head_dim != 256) return FA_ERR_UNSUPPORTED;
    const long long q_elems = (long long)batch * hq * sq * head_dim;
    if (q_elems >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    const DeviceInfo* di = device_info();
    if (!di) return FA_ERR_CUDA;
    if (!di->supported) return FA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (sk == 0)
        return from_cuda(launch_fill_empty(static_cast<uint16_t*>(o), lse,
                                           (long long)batch * hq * sq, head_dim, sinks, hq, sq,
                                           s));
    // several queries of a GQA group (contiguous caches, no window, the
    // library's own split count): the prefill kernel with the group's heads
    // packed into one tile
    if (num_splits <= 0 && block_table == nullptr && window <= 0 && head_dim == 128 &&
        (hq / hkv) * sq >= kDecodeToPrefillRows)
        return prefill_impl(q, k, v, o, lse, batch, hq, hkv, sq, sk, seqlens_k, head_dim, scale,
                            causal, 0, sinks, nullptr, 0, 0, 0, stream, nullptr);

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
    a.window = window > 0 ? window : 0;
    a.sinks = sinks;
    a.block_table = block_table;
    a.max_pages = max_pages;
    a.page_size = page_size;
    a.num_pages = num_pages;
    a.scale_log2 = scale * 1.4426950408889634f;
    if ((long long)hkv * a.n_mtiles > 65535) return FA_ERR_INVALID_ARG;
    // split planning: equal chunks of a multiple of 64 keys over the keys a
    // sequence's rows can see: all sk, or with a sliding window the last
    // window + sq - 1 (the splits start at each sequence's first visible key,
    // rounded down to a multiple of 64: up to 63 more)
    const long long span = a.window > 0 ? std::min<long long>(sk, (long long)a.window + sq + 62)
                                        : (long long)sk;
    int splits = num_splits;
    if (splits <= 0) {
        const long long pairs = (long long)batch * hkv * a.n_mtiles;
        const long long target = 24ll * di->num_sms;   // CTAs worth keeping in flight
        long long want = (target + pairs - 1) / pairs;
        const long long max_splits = (span + 255) / 256;  // at least 256 keys per split
        if (want > max_splits) want = max_splits;
        if (want < 1) want = 1;
        splits = (int)want;
    }
    long long chunk = (span + splits - 1) / splits;
    chunk = (chunk + 63) / 64 * 64;
    a.chunk = (int)chunk;
    a.n_splits = (int)((span + chunk - 1) / chunk);
    const size_t rows = (size_t)batch * hq * sq;
    const size_t bytes_o = (size_t)a.n_splits * rows * head_dim * sizeof(float);
    const size_t bytes_l = (size_t)a.n_splits * rows * sizeof(float);
    void* ws = nullptr;
    if (cudaMallocAsync(&ws, bytes_o + bytes_l, s) != cudaSuccess) return FA_ERR_CUDA;
    a.part_o = static_cast<float*>(ws);
    a.part_lse = reinterpret_cast<float*>(static_cast<char*>(ws) + bytes_o);
    cudaError_t e = launch_decode(a, head_dim, s);
    cudaError_t ef = cudaFreeAsync(ws, s);
    if (e != cudaSuccess || ef != cudaSuccess) return FA_ERR_CUDA;
    return FA_OK;
}

// Prefill on contiguous K/V (block_table == nullptr) or on paged caches
// [num_pages, hkv, page_size, d] (sk = max_pages * page_size keys per sequence).
// Packed variable-length sequences (see fa_fwd_prefill_varlen).
struct Varlen {
    const int* cu_seqlens_q;
    const int* cu_seqlens_k;
    int total_q, total_k;
};

// Dense, paged (block_table != nullptr) or packed (vl != nullptr; sq is then
// the largest query length and sk the largest key length) prefill.
fa_status prefill_impl(const void* q, const void* k, const void* v, void* o, float* lse, int batch,
                       int hq, int hkv, int sq, int sk, const int* seqlens_k, int head_dim,
                       float scale, int causal, int window, const float* sinks,
                       const int* block_table, int max_pages, int page_size, int num_pages,
                       fa_stream_t stream, const Varlen* vl = nullptr) {
    Common c;
    fa_status st = check_common(q, k, v, o, lse, batch, hq, hkv, sq, sk, scale, c);
    if (st != FA_OK || c.noop) return st;
    if ((reinterpret_cast<uintptr_t>(sinks) & 3u) != 0) return FA_ERR_MISALIGNED;
    if (!prefill_head_dim_ok(head_dim)) return FA_ERR_UNSUPPORTED;
    const DeviceInfo* di = device_info();
    if (!di) return FA_ERR_CUDA;
    if (!di->supported) return FA_ERR_UNSUPPORTED;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (sk == 0 || (vl && !block_table && vl->total_k == 0)) {
        // no keys anywhere: O = 0 and LSE = -inf (or the sink); for packed
        // sequences, O [total_q, hq, d] and LSE [hq, total_q] read as one
        // sequence of total_q rows
        const long long rows = vl ? (long long)vl->total_q * hq : (long long)batch * hq * sq;
        return from_cuda(launch_fill_empty(static_cast<uint16_t*>(o), lse, rows, head_dim, sinks,
                                           hq, vl ? vl->total_q : sq, s));
    }
    PrefillLaunch p{};
    const unsigned long long row_bytes = (unsigned long long)head_dim * 2;
    // kernel family, unit and block sizes, work split (head_dim 96 / 128,
    // dense and unmasked: the 256-key kernel)
    const PrefillShape shape = prefill_shape(batch, hq, sq, sk, head_dim, causal != 0, window,
                                             block_table != nullptr, vl != nullptr, di->num_sms,
                                             hq / hkv);
    const bool wide = shape.wide;
    // head-packed tiles: Q boxes of R rows x P heads, O boxes of 32 rows
    // (16 x 2 heads when R = 16)
    const unsigned pack_rows = (unsigned)shape.rows_per_unit;
    const unsigned o_box_rows = shape.pack > 1 && pack_rows < 32 ? pack_rows : 32;
    // Q, O: token-major packed tensors (map {d, tokens, heads}, a token's
    // heads adjacent) or dense [B, Hq, Sq, d]; K, V: paged caches, packed or
    // dense
    // (loads: prefill_load_map; the O store map is 3-D)
    if (vl) {
        if (!prefill_load_map(&p.tm_q, q, head_dim, vl->total_q, hq, row_bytes * hq, row_bytes) ||
            !encode_map_strided(&p.tm_o, o, head_dim, vl->total_q, hq, row_bytes * hq, row_bytes))
            return FA_ERR_INVALID_ARG;
    } else if (!(shape.pack > 1
                     ? encode_map_strided(&p.tm_q, q, head_dim, sq, (long long)batch * hq,
                                          row_bytes, row_bytes * sq, pack_rows,
                                          (unsigned)shape.pack)
                     : prefill_load_map(&p.tm_q, q, head_dim, sq, (long long)batch * hq,
                                        row_bytes, row_bytes * sq)) ||
               !encode_map(&p.tm_o, o, head_dim, sq, (long long)batch * hq) ||
               ((head_dim == 256 || wide) &&
                !encode_map32_strided(&p.tm_o32, o, head_dim, sq, (long long)batch * hq,
                                      row_bytes, row_bytes * sq, o_box_rows))) {
        return FA_ERR_INVALID_ARG;
    }
    if (block_table) {
        const long long planes = (long long)num_pages * hkv;
        if (!prefill_load_map(&p.tm_k, k, head_dim, page_size, planes, row_bytes,
                              row_bytes * page_size) ||
            !prefill_load_map(&p.tm_v, v, head_dim, page_size, planes, row_bytes,
                              row_bytes * page_size, true))
            return FA_ERR_INVALID_ARG;
    } else if (vl) {
        if (!prefill_load_map(&p.tm_k, k, head_dim, vl->total_k, hkv, row_bytes * hkv, row_bytes) ||
            !prefill_load_map(&p.tm_v, v, head_dim, vl->total_k, hkv, row_bytes * hkv, row_bytes,
                              true))
            return FA_ERR_INVALID_ARG;
    } else if (!(wide ? encode_map_strided(&p.tm_k, k, head_dim, sk, (long long)batch * hkv,
                                           row_bytes, row_bytes * sk, 256)
                      : prefill_load_map(&p.tm_k, k, head_dim, sk, (long long)batch * hkv,
                                         row_bytes, row_bytes * sk)) ||
               !prefill_load_map(&p.tm_v, v, head_dim, sk, (long long)batch * hkv, row_bytes,
                                 row_bytes * sk, true)) {
        return FA_ERR_INVALID_ARG;
    }
    PrefillArgs& a = p.args;
    if (vl) {
        a.cu_seqlens_q = vl->cu_seqlens_q;
        a.cu_seqlens_k = vl->cu_seqlens_k;
        a.total_q = vl->total_q;
        a.total_k = vl->total_k;
    }
    a.o = static_cast<uint16_t*>(o);
    a.lse = lse;
    a.seqlens_k = seqlens_k;
    a.err_word = di->err_word;
    a.B = batch;
    a.Hq = hq;
    a.Hkv = hkv;
    a.Sq = sq;
    a.Sk = sk;
    a.group = hq / hkv;
    a.num_mblk = shape.num_mblk;
    a.pack = shape.pack;
    a.scale_log2 = scale * 1.4426950408889634f;
    a.wait_limit_ns = kWaitLimitNs;
    // head_dim 256: the producer of each CTA also prefetches into L2 the Q
    // tiles of the CTA one wave later (+2.5 % on the causal GQA workload,
    // whose 2048 short units each start with a DRAM round trip of a 64 KB Q
    // tile; no gain measured at the other head dimensions)
    a.q_prefetch = head_dim == 256 ? di->num_sms : 0;
    a.window = window > 0 ? window : 0;
    a.sinks = sinks;
    a.block_table = block_table;
    a.max_pages = max_pages;
    a.page_size = page_size;
    a.trace = g_trace_buf;
    a.trace_block = g_trace_block;
    p.head_dim = head_dim;
    p.causal = causal ? 1 : 0;
    p.num_sms = di->num_sms;
    p.wide = wide ? 1 : 0;
    // work split: whole units, then the last partial wave's units in pieces
    const long long units = shape.units;
    if (units * prefill_ctas_per_unit(head_dim) >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    a.nk = shape.nk;
    const PrefillPlan plan = shape.plan;
    a.n_full = plan.n_full;
    a.split = plan.split;
    a.n_work = plan.n_full + plan.n_tail * plan.split;
    p.n_tail = plan.n_tail;
    void* ws = nullptr;
    if (plan.n_tail > 0) {
        const int nq = wide ? 1 : shape.rows_per_unit / 128;   // Q tiles of a unit
        const size_t pieces = (size_t)plan.n_tail * plan.split;
        const size_t part_o = pieces * nq * head_dim * 128 * sizeof(float);
        const size_t part_ml = pieces * nq * 2 * 128 * sizeof(float);
        const size_t counts = (size_t)plan.n_tail * sizeof(unsigned long long);
        if (cudaMallocAsync(&ws, part_o + part_ml + counts, s) != cudaSuccess) return FA_ERR_CUDA;
        a.part_o = static_cast<float*>(ws);
        a.part_ml = reinterpret_cast<float*>(static_cast<char*>(ws) + part_o);
        a.part_count =
            reinterpret_cast<unsigned long long*>(static_cast<char*>(ws) + part_o + part_ml);
        a.epoch = next_prefill_epoch();
    }
    cudaError_t e;
    switch (head_dim) {
        case 64: e = launch_prefill_d64(p, s); break;
        case 96: e = launch_prefill_d96(p, s); break;
        case 128: e = launch_prefill_d128(p, s); break;
        case 256: e = launch_prefill_d256(p, s); break;
        default: e = launch_prefill_d512(p, s); break;
    }
    if (ws != nullptr && cudaFreeAsync(ws, s) != cudaSuccess) return FA_ERR_CUDA;
    return from_cuda(e);
}

}  // namespace
}  // namespace fa

using namespace fa;

extern "C" {

fa_status fa_fwd_prefill_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                            int batch, int hq, int hkv, int sq, int sk, const int* seqlens_k,
                            int head_dim, float scale, int causal, int window,
                            const float* sinks, fa_stream_t stream) {
    return prefill_impl(q, k, v, o, lse, batch, hq, hkv, sq, sk, seqlens_k, head_dim, scale,
                        causal, window, sinks, nullptr, 0, 0, 0, stream);
}

fa_status fa_fwd_prefill(const void* q, const void* k, const void* v, void* o, float* lse,
                         int batch, int hq, int hkv, int sq, int sk, const int* seqlens_k,
                         int head_dim, float scale, int causal, fa_stream_t stream) {
    return prefill_impl(q, k, v, o, lse, batch, hq, hkv, sq, sk, seqlens_k, head_dim, scale,
                        causal, 0, nullptr, nullptr, 0, 0, 0, stream);
}

fa_status fa_fwd_prefill_paged(const void* q, const void* k_cache, const void* v_cache, void* o,
                               float* lse, int batch, int hq, int hkv, int sq,
                               const int* seqlens_k, const int* block_table, int max_pages,
                               int page_size, int num_pages, int head_dim, float scale,
                               int causal, fa_stream_t stream) {
    fa_status st = check_paged(seqlens_k, block_table, max_pages, page_size, num_pages, batch, hq,
                               sq);
    if (st != FA_OK) return st;
    if (page_size % 128 != 0) return FA_ERR_UNSUPPORTED;   // a key tile must fit a page
    return prefill_impl(q, k_cache, v_cache, o, lse, batch, hq, hkv, sq, max_pages * page_size,
                        seqlens_k, head_dim, scale, causal, 0, nullptr, block_table, max_pages,
                        page_size, num_pages, stream);
}

fa_status fa_fwd_prefill_varlen(const void* q, const void* k, const void* v, void* o, float* lse,
                                const int* cu_seqlens_q, const int* cu_seqlens_k, int batch,
                                int max_seqlen_q, int max_seqlen_k, int total_q, int total_k,
                                int hq, int hkv, int head_dim, float scale, int causal,
                                int window, const float* sinks, fa_stream_t stream) {
    if (batch < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || total_q < 0 || total_k < 0)
        return FA_ERR_INVALID_ARG;
    if (batch == 0 || total_q == 0 || hq == 0) return FA_OK;   // nothing to compute
    if (max_seqlen_q == 0 || (total_k > 0 && max_seqlen_k == 0)) return FA_ERR_INVALID_ARG;
    if (!cu_seqlens_q || !cu_seqlens_k) return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) != 0 ||
        (reinterpret_cast<uintptr_t>(cu_seqlens_k) & 3u) != 0)
        return FA_ERR_MISALIGNED;
    if ((long long)total_q * hq * head_dim >= (1ll << 40) ||
        (long long)total_k * hkv * head_dim >= (1ll << 40))
        return FA_ERR_INVALID_ARG;
    const Varlen vl{cu_seqlens_q, cu_seqlens_k, total_q, total_k};
    return prefill_impl(q, k, v, o, lse, batch, hq, hkv, max_seqlen_q,
                        total_k > 0 ? max_seqlen_k : 0, nullptr, head_dim, scale, causal, window,
                        sinks, nullptr, 0, 0, 0, stream, &vl);
}

fa_status fa_fwd_prefill_varlen_paged(const void* q, const void* k_cache, const void* v_cache,
                                      void* o, float* lse, const int* cu_seqlens_q,
                                      const int* seqlens_k, const int* block_table,
                                      int max_pages, int page_size, int num_pages, int batch,
                                      int max_seqlen_q, int total_q, int hq, int hkv,
                                      int head_dim, float scale, int causal, int window,
                                      const float* sinks, fa_stream_t stream) {
    if (batch < 0 || max_seqlen_q < 0 || total_q < 0) return FA_ERR_INVALID_ARG;
    if (batch == 0 || total_q == 0 || hq == 0) return FA_OK;   // nothing to compute
    if (max_seqlen_q == 0 || !cu_seqlens_q) return FA_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(cu_seqlens_q) & 3u) != 0) return FA_ERR_MISALIGNED;
    fa_status st = check_paged(seqlens_k, block_table, max_pages, page_size, num_pages, batch, hq,
                               max_seqlen_q);
    if (st != FA_OK) return st;
    if (page_size % 128 != 0) return FA_ERR_UNSUPPORTED;   // a key tile must fit a page
    if ((long long)total_q * hq * head_dim >= (1ll << 40)) return FA_ERR_INVALID_ARG;
    const Varlen vl{cu_seqlens_q, nullptr, total_q, 0};
    return prefill_impl(q, k_cache, v_cache, o, lse, batch, hq, hkv, max_seqlen_q,
                        max_pages * page_size, seqlens_k, head_dim, scale, causal, window, sinks,
                        block_table, max_pages, page_size, num_pages, stream, &vl);
}

fa_status fa_fwd_decode(const void* q, const void* k, const void* v, void* o, float* lse,
                        int batch, int hq, int hkv, int sq, int sk, const int* seqlens_k,
                        int head_dim, float scale, int causal, fa_stream_t stream) {
    return decode_impl(q, k, v, o, lse, batch, hq, hkv, sq, sk, seqlens_k, head_dim, scale,
                       causal, 0, nullptr, 0, stream);
}

fa_status fa_fwd_decode_ex(const void* q, const void* k, const void* v, void* o, float* lse,
                           int batch, int hq, int hkv, int sq, int sk, const int* seqlens_k,
                           int head_dim, float scale, int causal, int window, const float* sinks,
                           fa_stream_t stream) {
    return decode_impl(q, k, v, o, lse, batch, hq, hkv, sq, sk, seqlens_k, head_dim, scale,
                       causal, window, sinks, 0, stream);
}

fa_status fa_fwd_decode_paged(const void* q, const void* k_cache, const void* v_cache, void* o,
                              float* lse, int batch, int hq, int hkv, int sq,
                              const int* seqlens_k, const int* block_table, int max_pages,
                              int page_size, int num_pages, int head_dim, float scale, int causal,
                              fa_stream_t stream) {
    fa_status st = check_paged(seqlens_k, block_table, max_pages, page_size, num_pages, batch, hq,
                               sq);
    if (st != FA_OK) return st;
    return decode_impl(q, k_cache, v_cache, o, lse, batch, hq, hkv, sq, max_pages * page_size,
                       seqlens_k, head_dim, scale, causal, 0, nullptr, 0, stream, block_table,
                       max_pages, page_size, num_pages);
}

fa_status fa_fwd_decode_splits(const void* q, const void* k, const void* v, void* o, float* lse,
                               int batch, int hq, int hkv, int sq, int sk, const int* seqlens_k,
                               int head_dim, float scale, int causal, int num_splits,
                               fa_stream_t stream) {
    return decode_impl(q, k, v, o, lse, batch, hq, hkv, sq, sk, seqlens_k, head_dim, scale,
                       causal, 0, nullptr, num_splits, stream);
}

const char* fa_status_string(fa_status status) {
    switch (status) {
        case FA_OK: return "FA_OK";
        case FA_ERR_INVALID_ARG: return "FA_ERR_INVALID_ARG";
        case FA_ERR_UNSUPPORTED: return "FA_ERR_UNSUPPORTED";
        case FA_ERR_MISALIGNED: return "FA_ERR_MISALIGNED";
        case FA_ERR_CUDA: return "FA_ERR_CUDA";
        case FA_ERR_TIMEOUT: return "FA_ERR_TIMEOUT";
        default: return "FA_ERR_UNKNOWN";
    }
}

fa_status fa_get_device_error(fa_stream_t stream) {
    return fa_get_device_error_word(stream, nullptr);
}

fa_status fa_get_device_error_word(fa_stream_t stream, unsigned int* word_out) {
    if (word_out) *word_out = 0;
    const DeviceInfo* di = device_info();
    if (!di) return FA_ERR_CUDA;
    if (!di->supported) return FA_ERR_UNSUPPORTED;
    if (cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess)
        return FA_ERR_CUDA;
    unsigned int word = 0;
    if (cudaMemcpy(&word, di->err_word, sizeof word, cudaMemcpyDeviceToHost) != cudaSuccess)
        return FA_ERR_CUDA;
    if (word_out) *word_out = word;
    if (word != 0) {
        const unsigned int zero = 0;
        if (cudaMemcpy(di->err_word, &zero, sizeof zero, cudaMemcpyHostToDevice) != cudaSuccess)
            return FA_ERR_CUDA;
        return FA_ERR_TIMEOUT;
    }
    return FA_OK;
}

fa_status fa_selftest_wait_timeout(long long limit_ns, fa_stream_t stream) {
    const DeviceInfo* di = device_info();
    if (!di) return FA_ERR_CUDA;
    if (!di->supported) return FA_ERR_UNSUPPORTED;
    if (limit_ns < 1000) limit_ns = 1000;
    if (limit_ns > 1000000000ll) limit_ns = 1000000000ll;
    return from_cuda(launch_wait_timeout_selftest(di->err_word, (unsigned long long)limit_ns,
                                                  reinterpret_cast<cudaStream_t>(stream)));
}

fa_status fa_selftest_tmem_roundtrip(const float* in, float* out, fa_stream_t stream) {
    if (!in || !out) return FA_ERR_INVALID_ARG;
    const DeviceInfo* di = device_info();
    if (!di) return FA_ERR_CUDA;
    if (!di->supported) return FA_ERR_UNSUPPORTED;
    return from_cuda(launch_selftest_tmem_roundtrip(in, out, reinterpret_cast<cudaStream_t>(stream)));
}

fa_status fa_selftest_mma_tile(const void* a, const void* b, float* d, int mode, int kdim,
                               fa_stream_t stream) {
    if (!a || !b || !d) return FA_ERR_INVALID_ARG;
    if (mode == 1) kdim = 128;
    if (mode != 0 && mode != 1) return FA_ERR_INVALID_ARG;
    if (kdim != 64 && kdim != 128 && kdim != 256) return FA_ERR_INVALID_ARG;
    if (!aligned16(a) || !aligned16(b)) return FA_ERR_MISALIGNED;
    const DeviceInfo* di = device_info();
    if (!di) return FA_ERR_CUDA;
    if (!di->supported) return FA_ERR_UNSUPPORTED;
    return from_cuda(launch_selftest_mma_tile(static_cast<const uint16_t*>(a),
                                              static_cast<const uint16_t*>(b), d, mode, kdim,
                                              di->err_word, reinterpret_cast<cudaStream_t>(stream)));
}

fa_status fa_selftest_exp2_poly(const float* x, float* y, int n, fa_stream_t stream) {
    if (n < 0 || (n > 0 && (!x || !y))) return FA_ERR_INVALID_ARG;
    const DeviceInfo* di = device_info();
    if (!di) return FA_ERR_CUDA;
    if (!di->supported) return FA_ERR_UNSUPPORTED;
    return from_cuda(launch_selftest_exp2_poly(x, y, n, reinterpret_cast<cudaStream_t>(stream)));
}

fa_status fa_debug_prefill_trace(unsigned long long* buf, int block) {
    if (buf != nullptr && block < 0) return FA_ERR_INVALID_ARG;
    if (buf != nullptr && !FA_PREFILL_TRACE) return FA_ERR_UNSUPPORTED;
    g_trace_buf = buf;
    g_trace_block = block;
    return FA_OK;
}

fa_status fa_debug_prefill_plan_gqa(int batch, int hq, int hkv, int sq, int sk, int head_dim,
                                    int causal, int window, int paged, int packed, int num_sms,
                                    int* out) {
    if (!out || batch <= 0 || hq <= 0 || hkv <= 0 || hq % hkv != 0 || sq <= 0 || sk <= 0 ||
        batch > 65535 || hq > 65535 || num_sms < 1)
        return FA_ERR_INVALID_ARG;
    if (!prefill_head_dim_ok(head_dim)) return FA_ERR_INVALID_ARG;
    const PrefillShape sh = prefill_shape(batch, hq, sq, sk, head_dim, causal != 0, window,
                                          paged != 0, packed != 0, num_sms, hq / hkv);
    if (sh.units * prefill_ctas_per_unit(head_dim) >= (1ll << 31)) return FA_ERR_INVALID_ARG;
    out[0] = sh.plan.n_full;
    out[1] = sh.plan.n_tail;
    out[2] = sh.plan.split;
    out[3] = sh.rows_per_unit;
    out[4] = sh.keys_per_block;
    out[5] = sh.persistent ? 1 : 0;
    out[6] = sh.pack;
    return FA_OK;
}

fa_status fa_debug_prefill_plan_ex(int batch, int hq, int sq, int sk, int head_dim, int causal,
                                   int window, int paged, int packed, int num_sms, int* out) {
    if (!out) return FA_ERR_INVALID_ARG;
    int full[7];
    const fa_status st = fa_debug_prefill_plan_gqa(batch, hq, hq > 0 ? hq : 1, sq, sk, head_dim,
                                                   causal, window, paged, packed, num_sms, full);
    if (st != FA_OK) return st;
    for (int i = 0; i < 6; ++i) out[i] = full[i];
    return FA_OK;
}

fa_status fa_debug_prefill_plan(int batch, int hq, int sq, int sk, int head_dim, int causal,
                                int num_sms, int* out) {
    if (!out) return FA_ERR_INVALID_ARG;
    int full[6];
    const fa_status st =
        fa_debug_prefill_plan_ex(batch, hq, sq, sk, head_dim, causal, 0, 0, 0, num_sms, full);
    if (st != FA_OK) return st;
    out[0] = full[0];
    out[1] = full[1];
    out[2] = full[2];
    return FA_OK;
}

int fa_version(void) { return 300; }

}  // extern "C"
