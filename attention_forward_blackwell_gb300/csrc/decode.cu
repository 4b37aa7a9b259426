// Split-KV decode attention for sm_103a.
//
// Decode is bound by HBM bandwidth: every valid key and value row is read
// once, and with Hq/Hkv query heads per key/value head ("b200-flash-attention4-
// planner" E.7: explicit Q-head to KV-head mapping and reuse) each row feeds
// all heads of its group.  The method is the same streaming online softmax as
// prefill ("b200-flash-attention4-planner" A1); the key range is split into
// chunks so that enough CTAs stream concurrently, and the chunks are merged by
// their LSE ("STAGE_D.md": O = sum_i exp(lse_i) O_i / sum_i exp(lse_i), exact
// because the chunks cover disjoint key sets; "fa4-sm120-research" lists
// SplitKV among the features its kernels lack).
//
// decode_split_kernel: CTA = (key split, key/value head x 16-row query tile,
// batch entry), 4 warps.  The query rows of one key/value head (group heads x
// Sq queries) are packed onto the M = 16 dimension of the warp-level
// m16n8k16 bf16 MMA; S = Q K^T and O += P V run on the tensor cores, the row
// max / sum use quad shuffles.  Each warp streams its own 16-key slices
// (keys 16 w + 64 i of the split) through a 16-byte cp.async ring with zero
// fill past the split end, so no key beyond the sequence length is read.
// The four warps' states are merged in shared memory and the CTA writes one
// normalised partial (O_s, LSE_s in log2 units).
//
// decode_combine_kernel: one warp per query row merges its splits.
#include "common.cuh"
#include "ptx.cuh"

namespace fa {

namespace {

constexpr float kLn2f = 0.69314718055994530942f;
constexpr float kLog2ef = 1.44269504088896340736f;
constexpr float kRebase = 8.0f;   // lazy rebase threshold, log2 units

template <int D>
struct DecodeTraits {
    static constexpr int WARPS = 4;
    static constexpr int THREADS = WARPS * 32;
    static constexpr int KB = 16;                       // keys per warp step
    static constexpr int ROW = D * 2;                   // bytes per key row
    static constexpr int GRAN = D / 8;                  // 16-byte granules per row
    static constexpr int SLICE = KB * ROW;              // bytes of a 16-key K (or V) slice
    static constexpr int STAGES = (D == 256) ? 2 : (D == 128 ? 3 : 4);
    static constexpr int WARP_BYTES = STAGES * 2 * SLICE;
    static constexpr int MERGE_BYTES = WARPS * 16 * (D + 2) * 4;
    static constexpr int SMEM = (WARPS * WARP_BYTES > MERGE_BYTES) ? WARPS * WARP_BYTES
                                                                   : MERGE_BYTES;
    static constexpr int NT = D / 8;                    // n8 tiles of O
};

// byte offset of granule g of key row `key` inside a slice (XOR swizzle keeps
// the 8 rows read by one ldmatrix phase on distinct bank groups)
template <int D>
__device__ __forceinline__ uint32_t swz(int key, int g) {
    return (uint32_t)(key * DecodeTraits<D>::ROW + ((g ^ (key & 7)) << 4));
}

template <int D, bool PAGED>
__global__ void __launch_bounds__(DecodeTraits<D>::THREADS)
    decode_split_kernel(const DecodeArgs a) {
    using T = DecodeTraits<D>;
    extern __shared__ __align__(128) uint8_t smem[];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int split = blockIdx.x;
    const int hkv = blockIdx.y / a.n_mtiles;
    const int mt = blockIdx.y % a.n_mtiles;
    const int b = blockIdx.z;
    int L = a.Sk;
    if (a.seqlens_k != nullptr) L = max(0, min(a.seqlens_k[b], a.Sk));
    // splits start at the first key any query row of the sequence can see,
    // rounded down to a multiple of 64 (with a sliding window, the keys
    // before it are never read; the rounding keeps 16-key slices aligned)
    const int k_base = (a.window > 0) ? (max(0, L - a.Sq - a.window + 1) & ~63) : 0;
    const int k_lo = k_base + split * a.chunk;
    if (k_lo >= L) return;                       // nothing of this sequence here
    const int k_hi = min(k_lo + a.chunk, L);
    const int nblk = (k_hi - k_lo + T::KB - 1) / T::KB;
    const int my_blocks = nblk > warp ? (nblk - warp + T::WARPS - 1) / T::WARPS : 0;

    // query rows of this thread's fragment: rq0 = lane/4, rq1 = lane/4 + 8
    const int rbase = mt * 16;
    int qi[2];            // query index i (for causal), -1 if the row is padding
    int qoff[2];          // element offset of the row in q / o
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
        const int pr = rbase + (lane >> 2) + 8 * hrow;
        if (pr < a.rows) {
            const int g = pr / a.Sq, i = pr % a.Sq;
            qi[hrow] = i;
            qoff[hrow] = ((b * a.Hq + hkv * a.group + g) * a.Sq + i) * D;
        } else {
            qi[hrow] = -1;
            qoff[hrow] = -1;
        }
    }
    // Q as A fragments (row-major 16 x 16 per k-step)
    uint32_t qa[D / 16][4];
#pragma unroll
    for (int kk = 0; kk < D / 16; ++kk) {
        const int c0 = kk * 16 + 2 * (lane & 3);
#pragma unroll
        for (int hrow = 0; hrow < 2; ++hrow) {
            uint32_t lo = 0, hi = 0;
            if (qoff[hrow] >= 0) {
                lo = *reinterpret_cast<const uint32_t*>(a.q + qoff[hrow] + c0);
                hi = *reinterpret_cast<const uint32_t*>(a.q + qoff[hrow] + c0 + 8);
            }
            qa[kk][hrow] = lo;        // a0 (row lane/4) / a1 (row lane/4 + 8)
            qa[kk][2 + hrow] = hi;    // a2 / a3
        }
    }
    // last and first visible key per fragment row (bottom-right causal
    // alignment; sliding window)
    int lim[2], lo[2];
    int lo_min = 0x7fffffff;
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
        lim[hrow] = k_hi - 1;
        if (a.causal && qi[hrow] >= 0) lim[hrow] = min(lim[hrow], qi[hrow] + L - a.Sq);
        lo[hrow] = (a.window > 0 && qi[hrow] >= 0) ? qi[hrow] + L - a.Sq - a.window + 1 : 0;
        if (qi[hrow] >= 0) lo_min = min(lo_min, lo[hrow]);
    }
    // a split wholly below every row's window holds nothing for this tile;
    // the combine skips it for each row (it reads only splits that reach a
    // row's window)
    lo_min = min(lo_min, __shfl_xor_sync(0xffffffffu, lo_min, 4));
    lo_min = min(lo_min, __shfl_xor_sync(0xffffffffu, lo_min, 8));
    lo_min = min(lo_min, __shfl_xor_sync(0xffffffffu, lo_min, 16));
    if (k_hi <= lo_min) return;

    const uint32_t wbase = smem_u32(smem) + warp * T::WARP_BYTES;
    const size_t head_off = ((size_t)b * a.Hkv + hkv) * (size_t)a.Sk * D;
    // element offset of key row `key` of this sequence and key/value head
    auto row_off = [&](int key) -> size_t {
        if (!PAGED) return head_off + (size_t)key * D;
        int page = a.block_table[(size_t)b * a.max_pages + key / a.page_size];
        page = min(max(page, 0), a.num_pages - 1);
        return ((size_t)page * a.Hkv + hkv) * (size_t)a.page_size * D +
               (size_t)(key % a.page_size) * D;
    };

    // paged caches whose pages hold whole 16-key slices (slices start at
    // multiples of 16): one page lookup per slice instead of one per row
    const bool slice_pages = PAGED && a.page_size % T::KB == 0;

    auto load_block = [&](int i) {
        const int stage = i % T::STAGES;
        const int key0 = k_lo + T::KB * (warp + T::WARPS * i);
        const uint32_t sk = wbase + stage * 2 * T::SLICE;
        const uint32_t sv = sk + T::SLICE;
        const size_t slice_off = slice_pages ? row_off(key0) : 0;
#pragma unroll
        for (int e = lane; e < T::KB * T::GRAN; e += 32) {
            const int kr = e / T::GRAN, g = e % T::GRAN;
            const int key = key0 + kr;
            const bool valid = key < k_hi;
            const size_t src = (slice_pages ? slice_off + (size_t)(valid ? kr : 0) * D
                                            : row_off(valid ? key : k_lo)) + g * 8;
            cp_async_16(sk + swz<D>(kr, g), a.k + src, valid ? 16u : 0u);
            cp_async_16(sv + swz<D>(kr, g), a.v + src, valid ? 16u : 0u);
        }
    };

    float oacc[T::NT][4];
#pragma unroll
    for (int n = 0; n < T::NT; ++n) oacc[n][0] = oacc[n][1] = oacc[n][2] = oacc[n][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY};
    float l_run[2] = {0.f, 0.f};    // this thread's partial row sums
    const float sl2 = a.scale_log2;

#pragma unroll
    for (int s = 0; s < T::STAGES - 1; ++s) {
        if (s < my_blocks) load_block(s);
        cp_async_commit();
    }
    for (int i = 0; i < my_blocks; ++i) {
        cp_async_wait<T::STAGES - 2>();
        __syncwarp();
        const int stage = i % T::STAGES;
        const uint32_t sk = wbase + stage * 2 * T::SLICE;
        const uint32_t sv = sk + T::SLICE;
        const int key0 = k_lo + T::KB * (warp + T::WARPS * i);

        // S (16 rows x 16 keys) = Q K^T
        float sacc[2][4] = {{0.f, 0.f, 0.f, 0.f}, {0.f, 0.f, 0.f, 0.f}};
        {
            const int mi = lane >> 3, ri = lane & 7;
            const int key = (mi >> 1) * 8 + ri;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                uint32_t b00, b01, b10, b11;
                ldmatrix_x4(sk + swz<D>(key, 2 * kk + (mi & 1)), b00, b01, b10, b11);
                mma_bf16_16816(sacc[0], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b00, b01);
                mma_bf16_16816(sacc[1], qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3], b10, b11);
            }
        }
        // mask, running max (quad shuffle), lazy rebase
        float alpha[2];
        bool rebase = false;
#pragma unroll
        for (int hrow = 0; hrow < 2; ++hrow) {
            float mx = -INFINITY;
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int key = key0 + n * 8 + 2 * (lane & 3) + e;
                    float& sv_ = sacc[n][2 * hrow + e];
                    sv_ = (key <= lim[hrow] && key >= lo[hrow]) ? sv_ : -INFINITY;
                    mx = fmaxf(mx, sv_);
                }
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
            const float m_new = fmaxf(m_run[hrow], mx * sl2);
            alpha[hrow] = 1.f;
            if (m_new > m_run[hrow] + kRebase) {
                alpha[hrow] = ex2_approx(m_run[hrow] - m_new);
                m_run[hrow] = m_new;
                rebase = true;
            }
        }
        if (__any_sync(0xffffffffu, rebase)) {
#pragma unroll
            for (int n = 0; n < T::NT; ++n) {
                oacc[n][0] *= alpha[0];
                oacc[n][1] *= alpha[0];
                oacc[n][2] *= alpha[1];
                oacc[n][3] *= alpha[1];
            }
        }
        // P = exp2(s - m) as the A fragment of the value MMA
        uint32_t pa[4];
#pragma unroll
        for (int hrow = 0; hrow < 2; ++hrow) {
            const float base = (m_run[hrow] == -INFINITY) ? 0.f : m_run[hrow];
            float p[2][2];
#pragma unroll
            for (int n = 0; n < 2; ++n)
#pragma unroll
                for (int e = 0; e < 2; ++e) p[n][e] = ex2_approx(fmaf(sacc[n][2 * hrow + e], sl2, -base));
            l_run[hrow] = fmaf(l_run[hrow], alpha[hrow], (p[0][0] + p[0][1]) + (p[1][0] + p[1][1]));
            pa[hrow] = pack_bf16x2(p[0][0], p[0][1]);       // a0 / a1: keys 0..7
            pa[2 + hrow] = pack_bf16x2(p[1][0], p[1][1]);   // a2 / a3: keys 8..15
        }
        // O (16 rows x D) += P V
        {
            const int mi = lane >> 3, ri = lane & 7;
            const int key = (mi & 1) * 8 + ri;
#pragma unroll
            for (int nd = 0; nd < D / 16; ++nd) {
                uint32_t b0a, b1a, b0b, b1b;
                ldmatrix_x4_trans(sv + swz<D>(key, 2 * nd + (mi >> 1)), b0a, b1a, b0b, b1b);
                mma_bf16_16816(oacc[2 * nd], pa[0], pa[1], pa[2], pa[3], b0a, b1a);
                mma_bf16_16816(oacc[2 * nd + 1], pa[0], pa[1], pa[2], pa[3], b0b, b1b);
            }
        }
        __syncwarp();
        const int nxt = i + T::STAGES - 1;
        if (nxt < my_blocks) load_block(nxt);
        cp_async_commit();
    }
    cp_async_wait<0>();
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
        l_run[hrow] += __shfl_xor_sync(0xffffffffu, l_run[hrow], 1);
        l_run[hrow] += __shfl_xor_sync(0xffffffffu, l_run[hrow], 2);
    }
    __syncthreads();   // every warp is done with its ring; reuse it for the merge

    // merge the four warps: wm/wl [WARPS][16], wo [WARPS][16][D]
    float* wm = reinterpret_cast<float*>(smem);
    float* wl = wm + T::WARPS * 16;
    float* wo = wl + T::WARPS * 16;
#pragma unroll
    for (int hrow = 0; hrow < 2; ++hrow) {
        const int r = (lane >> 2) + 8 * hrow;
        if ((lane & 3) == 0) {
            wm[warp * 16 + r] = m_run[hrow];
            wl[warp * 16 + r] = l_run[hrow];
        }
#pragma unroll
        for (int n = 0; n < T::NT; ++n) {
            const int c = n * 8 + 2 * (lane & 3);
            wo[(warp * 16 + r) * D + c] = oacc[n][2 * hrow];
            wo[(warp * 16 + r) * D + c + 1] = oacc[n][2 * hrow + 1];
        }
    }
    __syncthreads();
    const int valid_rows = min(16, a.rows - rbase);
    for (int e = threadIdx.x; e < valid_rows * D; e += T::THREADS) {
        const int r = e / D, c = e % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < T::WARPS; ++w) M = fmaxf(M, wm[w * 16 + r]);
        const int pr = rbase + r;
        const int g = pr / a.Sq, qi_ = pr % a.Sq;
        const size_t row_id = ((size_t)b * a.Hq + hkv * a.group + g) * a.Sq + qi_;
        const size_t part = (size_t)split * a.B * a.Hq * a.Sq + row_id;
        float o = 0.f, lse2 = -INFINITY;
        if (M != -INFINITY) {
            float wsum = 0.f, acc = 0.f;
#pragma unroll
            for (int w = 0; w < T::WARPS; ++w) {
                const float f = ex2_approx(wm[w * 16 + r] - M);   // 0 for empty warps
                wsum = fmaf(f, wl[w * 16 + r], wsum);
                acc = fmaf(f, wo[(w * 16 + r) * D + c], acc);
            }
            o = acc / wsum;
            lse2 = M + lg2_approx(wsum);
        }
        a.part_o[part * D + c] = o;
        if (c == 0) a.part_lse[part] = lse2;
    }
}

// One warp per query row (b, hq, i): LSE-weighted merge of the splits that
// reach the row's keys, plus the row's attention sink (one more term of the
// normaliser without a value) if there is one.
template <int D>
__global__ void __launch_bounds__(256) decode_combine_kernel(const DecodeArgs a) {
    const int lane = threadIdx.x & 31;
    const long long row = (long long)blockIdx.x * 8 + (threadIdx.x >> 5);
    const long long n_rows = (long long)a.B * a.Hq * a.Sq;
    if (row >= n_rows) return;
    const int b = (int)(row / ((long long)a.Hq * a.Sq));
    const int h = (int)((row / a.Sq) % a.Hq);
    const int i = (int)(row % a.Sq);
    int L = a.Sk;
    if (a.seqlens_k != nullptr) L = max(0, min(a.seqlens_k[b], a.Sk));
    // the row's visible keys [k_first, k_last]
    int k_last = L - 1;
    if (a.causal) k_last = min(k_last, i + L - a.Sq);
    const int k_first = (a.window > 0) ? max(0, i + L - a.Sq - a.window + 1) : 0;
    // the splits start at the sequence's first visible key, rounded down to a
    // multiple of 64 (see the split kernel)
    const int k_base = (a.window > 0) ? (max(0, L - a.Sq - a.window + 1) & ~63) : 0;
    const int s_lo = (k_first - k_base) / a.chunk;
    const int ns = (k_last >= k_first) ? (L - k_base + a.chunk - 1) / a.chunk : 0;
    const size_t stride = (size_t)a.B * a.Hq * a.Sq;
    const float sg = (a.sinks != nullptr) ? a.sinks[h] * kLog2ef : -INFINITY;
    float M = sg;
    for (int s = s_lo; s < ns; ++s) M = fmaxf(M, a.part_lse[s * stride + row]);
    constexpr int PER = D / 32;
    float acc[PER];
#pragma unroll
    for (int e = 0; e < PER; ++e) acc[e] = 0.f;
    float wsum = 0.f;
    if (M != -INFINITY) {
        wsum = ex2_approx(sg - M);
        for (int s = s_lo; s < ns; ++s) {
            const float f = ex2_approx(a.part_lse[s * stride + row] - M);
            wsum += f;
            const float* po = a.part_o + (s * stride + row) * D;
#pragma unroll
            for (int e = 0; e < PER; ++e) acc[e] = fmaf(f, po[lane + 32 * e], acc[e]);
        }
    }
    const float inv = (wsum > 0.f) ? 1.f / wsum : 0.f;
    uint16_t* o = a.o + row * D;
#pragma unroll
    for (int e = 0; e < PER; ++e) {
        const uint32_t pk = pack_bf16x2(acc[e] * inv, 0.f);
        o[lane + 32 * e] = (uint16_t)(pk & 0xFFFFu);
    }
    if (lane == 0) a.lse[row] = (wsum > 0.f) ? (M + lg2_approx(wsum)) * kLn2f : -INFINITY;
}

template <int D>
cudaError_t launch_decode_impl(const DecodeArgs& a, cudaStream_t s) {
    using T = DecodeTraits<D>;
    void (*split)(DecodeArgs) =
        a.block_table != nullptr ? decode_split_kernel<D, true> : decode_split_kernel<D, false>;
    cudaError_t e = cudaFuncSetAttribute(split, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         T::SMEM);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)a.n_splits, (unsigned)(a.Hkv * a.n_mtiles), (unsigned)a.B);
    split<<<grid, T::THREADS, T::SMEM, s>>>(a);
    e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    const long long rows = (long long)a.B * a.Hq * a.Sq;
    decode_combine_kernel<D><<<(unsigned)((rows + 7) / 8), 256, 0, s>>>(a);
    return cudaGetLastError();
}

// ------------------------------------------------------ auxiliary kernels ----

// O = 0 and LSE = -inf (or the row's sink logit: the sink is then the only
// term of the softmax) for rows without any key.
__global__ void fill_empty_kernel(uint16_t* o, float* lse, long long rows, int d,
                                  const float* sinks, int hq, int sq) {
    const long long n = rows * d;
    for (long long e = (long long)blockIdx.x * blockDim.x + threadIdx.x; e < n;
         e += (long long)gridDim.x * blockDim.x) {
        o[e] = 0;
        if (e % d == 0) {
            const long long row = e / d;
            lse[row] = (sinks != nullptr) ? sinks[(row / sq) % hq] : -INFINITY;
        }
    }
}

// Waits on an mbarrier that nothing ever arrives at; the bounded wait gives up
// after limit_ns and records the time-out in the error word.
__global__ void wait_timeout_selftest_kernel(unsigned int* err_word, unsigned long long limit_ns) {
    __shared__ __align__(8) uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1);
        abort_flag = 0;
        mbar_fence_init();
    }
    __syncthreads();
    const WaitCtx wc{smem_u32(&abort_flag), (uint32_t)limit_ns, err_word};
    mbar_wait(smem_u32(&bar), 0, wc, kErrWaitTimeout | 0xFFu);
}

}  // namespace

cudaError_t launch_decode(const DecodeArgs& a, int head_dim, cudaStream_t s) {
    switch (head_dim) {
        case 64: return launch_decode_impl<64>(a, s);
        case 128: return launch_decode_impl<128>(a, s);
        case 256: return launch_decode_impl<256>(a, s);
        default: return cudaErrorInvalidValue;
    }
}

cudaError_t launch_fill_empty(uint16_t* o, float* lse, long long rows, int head_dim,
                              const float* sinks, int hq, int sq, cudaStream_t s) {
    if (rows <= 0) return cudaSuccess;
    long long blocks = (rows * head_dim + 255) / 256;
    if (blocks > 4096) blocks = 4096;
    fill_empty_kernel<<<(unsigned)blocks, 256, 0, s>>>(o, lse, rows, head_dim, sinks, hq, sq);
    return cudaGetLastError();
}

cudaError_t launch_wait_timeout_selftest(unsigned int* err_word, unsigned long long limit_ns,
                                         cudaStream_t s) {
    wait_timeout_selftest_kernel<<<1, 32, 0, s>>>(err_word, limit_ns);
    return cudaGetLastError();
}

}  // namespace fa
