// Warp-specialised prefill attention forward for sm_103a.
//
// Method: "b200-flash-attention4-planner".  Section A1 gives the streaming
// online softmax (per key/value block: S = Q K^T, new running max, rebase the
// old row_sum and O, P = exp(S - max), O += P V, divide by row_sum only at the
// end) and the role split (a TMA load warp, an MMA-issuing warp, softmax
// warpgroups for a two-stage Q pipeline, a correction/epilogue warpgroup, a
// store).  Section E steps 3-8 give the two MMAs, the S/P/O regions in tensor
// memory, the barrier graph (Q/K/V ready -> score MMA; S ready -> softmax;
// P ready + O safe -> value MMA; final O -> epilogue -> store), the scalar
// mailbox, the causal block classes (skipped / full / diagonal) and the O
// correction.  The design below is our own for sm_103a:
//
//   CTA = (query block, query head, batch entry).  For head_dim <= 128 a CTA
//   owns two 128-row Q tiles (NQ = 2) that share one K/V stream; for
//   head_dim = 256 it owns one Q tile (NQ = 1) and ping-pongs two score
//   buffers instead, because two 256-column O accumulators do not fit the
//   512 tensor-memory columns.
//
//   warps 0..4*NQ-1   softmax, one warpgroup per Q tile; thread = query row
//                     = tensor-memory lane
//   next warpgroup    correction (rebases O when the running max jumps) and
//                     epilogue (O / row_sum -> bf16 -> smem -> TMA store; LSE)
//   next warp         tcgen05.mma issue (one elected lane)
//   next warp         TMA producer (Q once, then K_j, V_j through the ring)
//
// Tensor memory (512 columns x 128 lanes x 32 bit):
//   NQ = 2: S_t at columns [128 t, 128 t + 128), O_t at [256 + 128 t, ...).
//           P_t (bf16 pairs) overwrites the upper half of S_t.
//   NQ = 1: S buffers at [0, 128) and [128, 256), O at [256, 512).
//
// Hazard on the P/S alias: the next score MMA S_t(j+1) overwrites the upper
// half of S_t, i.e. P_t(j), which the value MMA PV_t(j) reads.  The score MMA
// is therefore issued in two N=64 halves: the lower half (which never holds
// P) right after PV_t(j), the upper half only once PV_t(j) has completed
// (tcgen05.commit -> mbarrier).  Distinct-accumulator MMAs are not ordered by
// the ISA, so this wait is what makes the reuse safe; the lower-half MMA keeps
// the tensor core busy while the MMA warp waits.
//
// Rebasing: the running max m is only moved when the block max exceeds it by
// more than kRescaleThreshold (log2 units).  Until then P = exp2(s - m) may
// exceed 1 by at most 2^threshold, which fp32 accumulates exactly as well;
// O / row_sum and LSE = m + log2(row_sum) are unchanged by the choice of m.
// When m moves, both row_sum and O are multiplied by exp2(m_old - m_new), as
// the streaming recurrence requires.
#pragma once

#include "common.cuh"
#include "ptx.cuh"

namespace fa {

constexpr float kRescaleThreshold = 8.0f;   // log2 units (a factor of 256)
constexpr float kLn2 = 0.69314718055994530942f;

template <int D>
struct PrefillTraits {
    static constexpr int BM = 128;                     // rows per Q tile = TMEM lanes
    static constexpr int BN = 128;                     // keys per K/V tile
    static constexpr int NQ = (D <= 128) ? 2 : 1;      // Q tiles per CTA
    static constexpr int NSBUF = (NQ == 2) ? 1 : 2;    // score buffers per Q tile
    static constexpr int NCH = (D + 63) / 64;          // 64-element (128-byte) row chunks
    static constexpr int CHUNK = 128 * 128;            // one chunk of 128 rows, bytes
    static constexpr int QTILE = NCH * CHUNK;
    static constexpr int SLOT_CH = (NCH >= 2) ? 2 : 1; // chunks per ring slot
    static constexpr int PIECES = NCH / SLOT_CH;       // ring slots per K or V tile
    static constexpr int SLOT = SLOT_CH * CHUNK;
    static constexpr int NSLOT = (D == 64) ? 8 : 4;
    static constexpr int KSTEPS = D / 16;              // score MMA steps of K = 16
    static constexpr int D_COLS = D;                   // O accumulator columns
    // Value MMA N per instruction.  head_dim 96 runs N = 128: its second
    // 64-column V chunk is half zero-filled by TMA (columns past d read as
    // zero), so O columns 96..127 stay zero and are never stored.
    static constexpr int PV_N = (D == 96) ? 128 : ((D <= 128) ? D : 128);
    static constexpr int NUM_WARPS = (NQ + 2) * 4;
    static constexpr int THREADS = NUM_WARPS * 32;
    static constexpr int CORR_WG = NQ;
    static constexpr int MMA_WARP = (NQ + 1) * 4;
    static constexpr int LOAD_WARP = MMA_WARP + 1;
    static constexpr uint32_t TMEM_COLS = 512;
    // Register split (threads x registers after setmaxnreg must not exceed
    // the launch allocation: 512 x 128 for NQ = 2, 384 x 168 for NQ = 1).
    static constexpr uint32_t REG_SOFTMAX = (NQ == 2) ? 176 : 240;
    static constexpr uint32_t REG_CORR = (NQ == 2) ? 80 : 88;
    static constexpr uint32_t REG_OTHER = (NQ == 2) ? 80 : 80;
    static constexpr int SMEM_Q = NQ * QTILE;
    static constexpr int SMEM_RING = NSLOT * SLOT;
    static constexpr int SMEM_AUX = 4096;
    static constexpr int SMEM_TOTAL = 1024 + SMEM_Q + SMEM_RING + SMEM_AUX;

    __device__ static constexpr uint32_t s_col(int i) { return (uint32_t)(i * 128); }
    __device__ static constexpr uint32_t o_col(int t) {
        return (NQ == 2) ? (uint32_t)(256 + t * 128) : 256u;
    }
};

template <class T>
struct PrefillAux {
    uint64_t bar_q;
    uint64_t bar_full[T::NSLOT];
    uint64_t bar_empty[T::NSLOT];
    uint64_t bar_s_full[2];        // NQ = 2: per tile; NQ = 1: per score buffer
    uint64_t bar_p_ready[T::NQ];
    uint64_t bar_o_ready[T::NQ];
    uint64_t bar_pv_done[T::NQ];
    uint64_t bar_mb_full[T::NQ];
    uint64_t bar_mb_empty[T::NQ];
    uint64_t bar_epi[T::NQ];       // staging of O_t in shared memory complete
    uint64_t bar_drain;
    uint32_t tmem_base;
    int abort_flag;
    float mb_alpha[T::NQ][128];
    float mb_l[T::NQ][128];
    float mb_m[T::NQ][128];
};

// Wait-site codes (recorded with kErrWaitTimeout on a time-out).
enum : unsigned int {
    kSiteLoadEmpty = 1, kSiteMmaQ, kSiteMmaK, kSiteMmaV, kSiteMmaP, kSiteMmaO, kSiteMmaPv,
    kSiteSmS, kSiteSmMbox, kSiteCorrMbox, kSiteCorrPv, kSiteEpiMbox, kSiteEpiPv,
    kSiteEpiStage
};

// Per-CTA work coordinates, computed identically by every thread.
struct PrefillWork {
    int b, h, hk, row0, L, off;
    int n_kv[2];   // K/V tiles visited by Q tile 0 / 1
    int n_max;
};

template <class T, bool CAUSAL>
__device__ __forceinline__ PrefillWork prefill_work(const PrefillArgs& a) {
    PrefillWork w;
    const int mblk = CAUSAL ? (a.num_mblk - 1 - (int)blockIdx.x) : (int)blockIdx.x;
    w.h = blockIdx.y;
    w.b = blockIdx.z;
    w.hk = w.h / a.group;
    int L = a.Sk;
    if (a.seqlens_k != nullptr) L = max(0, min(a.seqlens_k[w.b], a.Sk));
    w.L = L;
    w.off = L - a.Sq;
    w.row0 = mblk * T::NQ * T::BM;
    w.n_kv[0] = w.n_kv[1] = 0;
#pragma unroll
    for (int t = 0; t < T::NQ; ++t) {
        int last = L - 1;   // last key any row of the tile can see
        if (CAUSAL) last = min(last, w.row0 + (t + 1) * T::BM - 1 + w.off);
        w.n_kv[t] = last >= 0 ? last / T::BN + 1 : 0;
    }
    w.n_max = w.n_kv[T::NQ - 1];
    return w;
}

// Ring position p (K_j piece c at p = 2 j PIECES + c, V_j at (2 j + 1) PIECES + c).
template <class T>
__device__ __forceinline__ uint32_t ring_slot(int p) { return (uint32_t)(p % T::NSLOT); }
template <class T>
__device__ __forceinline__ uint32_t ring_phase(int p) { return (uint32_t)((p / T::NSLOT) & 1); }

// ------------------------------------------------------------ producer ----

template <class T>
__device__ void prefill_load_role(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                                  const CUtensorMap* tm_v, const PrefillArgs& a,
                                  const PrefillWork& w, PrefillAux<T>* aux, uint32_t sQ,
                                  uint32_t sRing, const WaitCtx& wc) {
    const int lane = threadIdx.x & 31;
    if (w.n_max <= 0) return;
    const uint32_t bar_q = smem_u32(&aux->bar_q);
    if (lane == 0) {
        tma_prefetch_desc(tm_q);
        tma_prefetch_desc(tm_k);
        tma_prefetch_desc(tm_v);
        mbar_arrive_expect_tx(bar_q, (uint32_t)(T::NQ * T::QTILE));
#pragma unroll
        for (int t = 0; t < T::NQ; ++t)
#pragma unroll
            for (int c = 0; c < T::NCH; ++c)
                tma_load_3d(sQ + t * T::QTILE + c * T::CHUNK, tm_q, c * 64, w.row0 + t * T::BM,
                            w.b * a.Hq + w.h, bar_q);
    }
    int issued = 0;
    const int total = 2 * w.n_max * T::PIECES;
    for (int p = 0; p < total; ++p) {
        const int j = p / (2 * T::PIECES);
        const int kv = (p / T::PIECES) & 1;
        const int pc = p % T::PIECES;
        const uint32_t slot = ring_slot<T>(p);
        if (!mbar_wait(smem_u32(&aux->bar_empty[slot]), ring_phase<T>(p) ^ 1u, wc,
                       kErrWaitTimeout | kSiteLoadEmpty))
            break;
        if (lane == 0) {
            const uint32_t full = smem_u32(&aux->bar_full[slot]);
            mbar_arrive_expect_tx(full, (uint32_t)T::SLOT);
            const CUtensorMap* m = kv ? tm_v : tm_k;
#pragma unroll
            for (int c = 0; c < T::SLOT_CH; ++c)
                tma_load_3d(sRing + slot * T::SLOT + c * T::CHUNK, m, (pc * T::SLOT_CH + c) * 64,
                            j * T::BN, w.b * a.Hkv + w.hk, full);
        }
        __syncwarp();
        issued = p + 1;
    }
    // Drain: every copy issued by this warp must have landed before the CTA
    // exits (on the normal path they all have; after an abort some may not).
    if (lane == 0) {
        mbar_wait_drain(bar_q, 0, a.wait_limit_ns);
        const int first = issued > T::NSLOT ? issued - T::NSLOT : 0;
        for (int p = first; p < issued; ++p)
            mbar_wait_drain(smem_u32(&aux->bar_full[ring_slot<T>(p)]), ring_phase<T>(p),
                            a.wait_limit_ns);
    }
    __syncwarp();
}

// ----------------------------------------------------------- MMA issue ----

// Zeroes value rows [rv, BN) of a K/V tile held in ring slots starting at
// position p (rows past the sequence length; they may hold anything, and a
// zero probability times a non-finite value would poison O).
template <class T>
__device__ __forceinline__ void zero_value_tail(uint32_t sRing, int p, int rv) {
    const int lane = threadIdx.x & 31;
    const int granules = (T::BN - rv) * 8;   // 16-byte granules per chunk
#pragma unroll
    for (int pc = 0; pc < T::PIECES; ++pc) {
        const uint32_t slot = ring_slot<T>(p + pc);
#pragma unroll
        for (int c = 0; c < T::SLOT_CH; ++c) {
            const uint32_t base = sRing + slot * T::SLOT + c * T::CHUNK + rv * 128;
            for (int g = lane; g < granules; g += 32)
                asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(base + g * 16),
                             "r"(0)
                             : "memory");
        }
    }
    fence_proxy_async_smem();
    __syncwarp();
}

// Score MMA S[cols] = Q_t * K^T over all head dims, for K rows [64 hf, 64 hf + n).
template <class T>
__device__ __forceinline__ void issue_score(uint32_t tmem_d, uint32_t sQt, uint32_t sRing,
                                            int posK, int hf, uint32_t idesc) {
#pragma unroll
    for (int kk = 0; kk < T::KSTEPS; ++kk) {
        const int piece = kk / (T::SLOT_CH * 4);
        const int ch = (kk / 4) % T::SLOT_CH;
        const uint32_t a_addr = sQt + (kk / 4) * T::CHUNK + (kk % 4) * 32;
        const uint32_t b_addr = sRing + ring_slot<T>(posK + piece) * T::SLOT + ch * T::CHUNK +
                                hf * 64 * 128 + (kk % 4) * 32;
        umma_ss(tmem_d, sdesc_sw128(a_addr, 16, 1024), sdesc_sw128(b_addr, 16, 1024), idesc,
                kk > 0 ? 1u : 0u);
    }
}

// Value MMA O[:, n-half] (+)= P * V over 128 keys (8 steps of 16 keys).
template <class T>
__device__ __forceinline__ void issue_value(uint32_t tmem_o, uint32_t tmem_p, uint32_t v_slot_addr,
                                            uint32_t idesc, bool first) {
#pragma unroll
    for (int kk = 0; kk < T::BN / 16; ++kk) {
        const uint64_t bd = sdesc_sw128(v_slot_addr + kk * 2048, T::CHUNK, 1024);
        umma_ts(tmem_o, tmem_p + kk * 8, bd, idesc, (!first || kk > 0) ? 1u : 0u);
    }
}

template <class T>
__device__ void prefill_mma_role(const PrefillArgs& a, const PrefillWork& w, PrefillAux<T>* aux,
                                 uint32_t tmem, uint32_t sQ, uint32_t sRing, const WaitCtx& wc) {
    const int lane = threadIdx.x & 31;
    const bool leader = lane == 0;
    auto full_bar = [&](int p) { return smem_u32(&aux->bar_full[ring_slot<T>(p)]); };
    auto empty_bar = [&](int p) { return smem_u32(&aux->bar_empty[ring_slot<T>(p)]); };
    auto wait_tile = [&](int p0, unsigned site) {
        for (int pc = 0; pc < T::PIECES; ++pc)
            if (!mbar_wait(full_bar(p0 + pc), ring_phase<T>(p0 + pc), wc, kErrWaitTimeout | site))
                return false;
        return true;
    };
    auto release_tile = [&](int p0) {
        if (leader)
            for (int pc = 0; pc < T::PIECES; ++pc) tc_commit(empty_bar(p0 + pc));
    };

    if (w.n_max > 0) do {
        if (!mbar_wait(smem_u32(&aux->bar_q), 0, wc, kErrWaitTimeout | kSiteMmaQ)) break;
        if (!wait_tile(0, kSiteMmaK)) break;
        tc_fence_after();
        bool ok = true;
        if constexpr (T::NQ == 2) {
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, 64, false, false);
            constexpr uint32_t idesc_v = idesc_bf16_f32(128, T::PV_N, false, true);
            if (leader) {
                for (int t = 0; t < 2; ++t) {
                    if (w.n_kv[t] <= 0) continue;
                    issue_score<T>(tmem + T::s_col(t), sQ + t * T::QTILE, sRing, 0, 0, idesc_s);
                    issue_score<T>(tmem + T::s_col(t) + 64, sQ + t * T::QTILE, sRing, 0, 1, idesc_s);
                    tc_commit(smem_u32(&aux->bar_s_full[t]));
                }
            }
            release_tile(0);
            __syncwarp();
            for (int j = 0; j < w.n_max && ok; ++j) {
                const int posV = (2 * j + 1) * T::PIECES;
                const int posK = (2 * j + 2) * T::PIECES;
                if (!wait_tile(posV, kSiteMmaV)) { ok = false; break; }
                if (j == w.n_max - 1 && w.L - j * T::BN < T::BN)
                    zero_value_tail<T>(sRing, posV, w.L - j * T::BN);
                bool k_next_ready = false;
                for (int t = 0; t < 2; ++t) {
                    if (j >= w.n_kv[t]) continue;
                    const uint32_t ph = (uint32_t)(j & 1);
                    if (!mbar_wait(smem_u32(&aux->bar_p_ready[t]), ph, wc, kErrWaitTimeout | kSiteMmaP) ||
                        !mbar_wait(smem_u32(&aux->bar_o_ready[t]), ph, wc, kErrWaitTimeout | kSiteMmaO)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (leader) {
                        issue_value<T>(tmem + T::o_col(t), tmem + T::s_col(t) + 64,
                                       sRing + ring_slot<T>(posV) * T::SLOT, idesc_v, j == 0);
                        tc_commit(smem_u32(&aux->bar_pv_done[t]));
                        if (t == 1) tc_commit(empty_bar(posV));   // V_j fully consumed
                    }
                    __syncwarp();
                    if (j + 1 < w.n_kv[t]) {
                        if (!k_next_ready) {
                            if (!wait_tile(posK, kSiteMmaK)) { ok = false; break; }
                            k_next_ready = true;
                            tc_fence_after();
                        }
                        if (leader)
                            issue_score<T>(tmem + T::s_col(t), sQ + t * T::QTILE, sRing, posK, 0,
                                           idesc_s);
                        __syncwarp();
                        // the upper half overwrites P_t(j): wait until PV_t(j) is done
                        if (!mbar_wait(smem_u32(&aux->bar_pv_done[t]), ph, wc,
                                       kErrWaitTimeout | kSiteMmaPv)) {
                            ok = false;
                            break;
                        }
                        tc_fence_after();
                        if (leader) {
                            issue_score<T>(tmem + T::s_col(t) + 64, sQ + t * T::QTILE, sRing, posK,
                                           1, idesc_s);
                            tc_commit(smem_u32(&aux->bar_s_full[t]));
                        }
                        __syncwarp();
                    }
                }
                if (ok && j + 1 < w.n_max) release_tile(posK);
                __syncwarp();
            }
        } else {
            constexpr uint32_t idesc_s = idesc_bf16_f32(128, 128, false, false);
            constexpr uint32_t idesc_v = idesc_bf16_f32(128, T::PV_N, false, true);
            if (leader) {
                issue_score<T>(tmem + T::s_col(0), sQ, sRing, 0, 0, idesc_s);
                tc_commit(smem_u32(&aux->bar_s_full[0]));
            }
            release_tile(0);
            __syncwarp();
            for (int j = 0; j < w.n_max; ++j) {
                const int posV = (2 * j + 1) * T::PIECES;
                const int posK = (2 * j + 2) * T::PIECES;
                if (j + 1 < w.n_max) {
                    if (!wait_tile(posK, kSiteMmaK)) { ok = false; break; }
                    // buffer (j+1)%2 held P(j-1): PV(j-1) must have completed
                    if (j >= 1 && !mbar_wait(smem_u32(&aux->bar_pv_done[0]), (uint32_t)((j - 1) & 1),
                                             wc, kErrWaitTimeout | kSiteMmaPv)) {
                        ok = false;
                        break;
                    }
                    tc_fence_after();
                    if (leader) {
                        issue_score<T>(tmem + T::s_col((j + 1) & 1), sQ, sRing, posK, 0, idesc_s);
                        tc_commit(smem_u32(&aux->bar_s_full[(j + 1) & 1]));
                    }
                    release_tile(posK);
                    __syncwarp();
                }
                if (!wait_tile(posV, kSiteMmaV)) { ok = false; break; }
                if (j == w.n_max - 1 && w.L - j * T::BN < T::BN)
                    zero_value_tail<T>(sRing, posV, w.L - j * T::BN);
                const uint32_t ph = (uint32_t)(j & 1);
                if (!mbar_wait(smem_u32(&aux->bar_p_ready[0]), ph, wc, kErrWaitTimeout | kSiteMmaP) ||
                    !mbar_wait(smem_u32(&aux->bar_o_ready[0]), ph, wc, kErrWaitTimeout | kSiteMmaO)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
                if (leader) {
#pragma unroll
                    for (int nh = 0; nh < T::PIECES; ++nh)
                        issue_value<T>(tmem + T::o_col(0) + nh * 128, tmem + T::s_col(j & 1) + 64,
                                       sRing + ring_slot<T>(posV + nh) * T::SLOT, idesc_v, j == 0);
                    tc_commit(smem_u32(&aux->bar_pv_done[0]));
                }
                release_tile(posV);
                __syncwarp();
            }
        }
    } while (0);
    // All MMAs of this CTA must have completed before tensor memory is freed.
    if (leader) {
        tc_commit(smem_u32(&aux->bar_drain));
        mbar_wait_drain(smem_u32(&aux->bar_drain), 0, a.wait_limit_ns);
    }
    __syncwarp();
}

// ------------------------------------------------------------- softmax ----

template <class T, bool CAUSAL>
__device__ void prefill_softmax_role(int t, const PrefillArgs& a, const PrefillWork& w,
                                     PrefillAux<T>* aux, uint32_t tmem, const WaitCtx& wc) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = (warp & 3) * 32 + lane;                    // tile row = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int row = w.row0 + t * T::BM + r;
    int lim = w.L - 1;                                       // last visible key of this row
    if (CAUSAL) lim = min(lim, row + w.off);
    const float sl2 = a.scale_log2;
    const int nk = w.n_kv[t];
    float m_run = -INFINITY;   // running max of scaled scores, log2 units (the basis)
    float l_run = 0.f;         // running row_sum in that basis
    const uint32_t mb_full = smem_u32(&aux->bar_mb_full[t]);
    const uint32_t mb_empty = smem_u32(&aux->bar_mb_empty[t]);
    bool ok = true;
    for (int j = 0; j < nk; ++j) {
        const int sb = (T::NSBUF == 2) ? (j & 1) : 0;
        const uint32_t scol = (T::NQ == 2) ? T::s_col(t) : T::s_col(sb);
        const uint32_t bar_s = smem_u32(&aux->bar_s_full[(T::NQ == 2) ? t : sb]);
        const uint32_t par_s = (T::NQ == 2) ? (uint32_t)(j & 1) : (uint32_t)((j >> 1) & 1);
        if (!mbar_wait(bar_s, par_s, wc, kErrWaitTimeout | kSiteSmS)) { ok = false; break; }
        tc_fence_after();
        uint32_t u[4][32];
#pragma unroll
        for (int q = 0; q < 4; ++q) tmem_ld32(lane_base + scol + q * 32, u[q]);
        tmem_wait_ld();
        float s[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(u[c >> 5][c & 31]);
        // mask: only tiles that reach past this row's last visible key
        const int kv0 = j * T::BN;
        if (lim - kv0 < T::BN - 1) {
            const int nvis = lim - kv0 + 1;                  // visible columns (may be <= 0)
#pragma unroll
            for (int c = 0; c < 128; ++c) s[c] = (c < nvis) ? s[c] : -INFINITY;
        }
        float mx = fmax3(s[0], s[1], s[2]);
#pragma unroll
        for (int c = 3; c < 127; c += 2) mx = fmax3(mx, s[c], s[c + 1]);
        mx = fmaxf(mx, s[127]);
        const float m_new = fmaxf(m_run, mx * sl2);
        float alpha = 1.f;
        if (m_new > m_run + kRescaleThreshold) {
            alpha = ex2_approx(m_run - m_new);   // 0 when m_run = -inf
            m_run = m_new;
        }
        // mailbox message j: the rebase factor, for the correction warpgroup
        if (!mbar_wait(mb_empty, (uint32_t)((j & 1) ^ 1), wc, kErrWaitTimeout | kSiteSmMbox)) {
            ok = false;
            break;
        }
        aux->mb_alpha[t][r] = alpha;
        mbar_arrive(mb_full);
        const float base = (m_run == -INFINITY) ? 0.f : m_run;
        float rs0 = 0.f, rs1 = 0.f;
        uint32_t pk[2][32];
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            const float p0 = ex2_approx(fmaf(s[2 * c], sl2, -base));
            const float p1 = ex2_approx(fmaf(s[2 * c + 1], sl2, -base));
            rs0 += p0;
            rs1 += p1;
            pk[c >> 5][c & 31] = pack_bf16x2(p0, p1);
        }
        l_run = fmaf(l_run, alpha, rs0 + rs1);
        tmem_st32(lane_base + scol + 64, pk[0]);
        tmem_st32(lane_base + scol + 96, pk[1]);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive(smem_u32(&aux->bar_p_ready[t]));
    }
    if (ok) {   // final message nk: row statistics for the epilogue
        if (mbar_wait(mb_empty, (uint32_t)((nk & 1) ^ 1), wc, kErrWaitTimeout | kSiteSmMbox)) {
            aux->mb_l[t][r] = l_run;
            aux->mb_m[t][r] = m_run;
            mbar_arrive(mb_full);
        }
    }
}

// ---------------------------------------------------- correction/epilogue ----

template <class T>
__device__ void prefill_correction_role(const CUtensorMap* tm_o, const PrefillArgs& a,
                                        const PrefillWork& w, PrefillAux<T>* aux, uint32_t tmem,
                                        uint32_t sQ, const WaitCtx& wc) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const bool issuer = (warp & 3) == 0 && lane == 0;
    bool ok = true;
    for (int j = 0; j < w.n_max && ok; ++j) {
        for (int t = 0; t < T::NQ; ++t) {
            if (j >= w.n_kv[t]) continue;
            if (!mbar_wait(smem_u32(&aux->bar_mb_full[t]), (uint32_t)(j & 1), wc,
                           kErrWaitTimeout | kSiteCorrMbox)) {
                ok = false;
                break;
            }
            const float alpha = aux->mb_alpha[t][r];
            mbar_arrive(smem_u32(&aux->bar_mb_empty[t]));
            if (j > 0 && __any_sync(0xffffffffu, alpha < 1.f)) {
                // O_t must hold PV_t(j-1) before it is rebased
                if (!mbar_wait(smem_u32(&aux->bar_pv_done[t]), (uint32_t)((j - 1) & 1), wc,
                               kErrWaitTimeout | kSiteCorrPv)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
#pragma unroll 1
                for (int c = 0; c < T::D_COLS / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld32(lane_base + T::o_col(t) + c * 32, v);
                    tmem_wait_ld();
#pragma unroll
                    for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                    tmem_st32(lane_base + T::o_col(t) + c * 32, v);
                }
                tmem_wait_st();
            }
            tc_fence_before();
            mbar_arrive(smem_u32(&aux->bar_o_ready[t]));
        }
    }
    // epilogue: O / row_sum -> bf16 -> shared (Q tile's space, 128-byte swizzled) -> TMA store
    for (int t = 0; t < T::NQ && ok; ++t) {
        const int nk = w.n_kv[t];
        if (!mbar_wait(smem_u32(&aux->bar_mb_full[t]), (uint32_t)(nk & 1), wc,
                       kErrWaitTimeout | kSiteEpiMbox)) {
            ok = false;
            break;
        }
        const float l = aux->mb_l[t][r];
        const float m = aux->mb_m[t][r];
        if (nk > 0) {
            if (!mbar_wait(smem_u32(&aux->bar_pv_done[t]), (uint32_t)((nk - 1) & 1), wc,
                           kErrWaitTimeout | kSiteEpiPv)) {
                ok = false;
                break;
            }
            tc_fence_after();
        }
        const float inv_l = (l > 0.f) ? 1.f / l : 0.f;
        const uint32_t stage = sQ + t * T::QTILE;
#pragma unroll 1
        for (int c32 = 0; c32 < (T::D_COLS + 31) / 32; ++c32) {
            uint32_t v[32];
            if (nk > 0) {
                tmem_ld32(lane_base + T::o_col(t) + c32 * 32, v);
                tmem_wait_ld();
            } else {
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = 0u;
            }
            const int ch = c32 >> 1;                 // 64-column chunk
            const uint32_t row_addr = stage + ch * T::CHUNK + r * 128;
#pragma unroll
            for (int g4 = 0; g4 < 4; ++g4) {
                const int g = (c32 & 1) * 4 + g4;    // 16-byte granule within the 128-byte row
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e)
                    pk[e] = pack_bf16x2(__uint_as_float(v[g4 * 8 + 2 * e]) * inv_l,
                                        __uint_as_float(v[g4 * 8 + 2 * e + 1]) * inv_l);
                const uint32_t addr = row_addr + ((uint32_t)(g ^ (r & 7)) << 4);
                asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[0]),
                             "r"(pk[1]), "r"(pk[2]), "r"(pk[3])
                             : "memory");
            }
        }
        const int row = w.row0 + t * T::BM + r;
        if (row < a.Sq) {
            const float lse = (l > 0.f) ? (m + lg2_approx(l)) * kLn2 : -INFINITY;
            a.lse[((size_t)w.b * a.Hq + w.h) * a.Sq + row] = lse;
        }
        fence_proxy_async_smem();
        mbar_arrive(smem_u32(&aux->bar_epi[t]));
        if (issuer && w.row0 + t * T::BM < a.Sq &&
            mbar_wait_lane(smem_u32(&aux->bar_epi[t]), 0, wc, kErrWaitTimeout | kSiteEpiStage)) {
#pragma unroll
            for (int ch = 0; ch < T::NCH; ++ch)
                tma_store_3d(tm_o, stage + ch * T::CHUNK, ch * 64, w.row0 + t * T::BM,
                             w.b * a.Hq + w.h);
            bulk_commit_group();
        }
    }
    if (issuer) bulk_wait_group_0();
}

// --------------------------------------------------------------- kernel ----

template <int D, bool CAUSAL>
__global__ void __launch_bounds__(PrefillTraits<D>::THREADS, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                   const PrefillArgs args) {
    using T = PrefillTraits<D>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sQ = (raw + 1023u) & ~1023u;   // 1024-aligned: swizzle atoms
    const uint32_t sRing = sQ + T::SMEM_Q;
    auto* aux = reinterpret_cast<PrefillAux<T>*>(smem_raw + (sQ - raw) + T::SMEM_Q + T::SMEM_RING);

    const int warp = threadIdx.x >> 5;
    const int wg = warp >> 2;
    const PrefillWork w = prefill_work<T, CAUSAL>(args);

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&aux->bar_q), 1);
        for (int i = 0; i < T::NSLOT; ++i) {
            mbar_init(smem_u32(&aux->bar_full[i]), 1);
            mbar_init(smem_u32(&aux->bar_empty[i]), 1);
        }
        for (int i = 0; i < 2; ++i) mbar_init(smem_u32(&aux->bar_s_full[i]), 1);
        for (int t = 0; t < T::NQ; ++t) {
            mbar_init(smem_u32(&aux->bar_p_ready[t]), 128);
            mbar_init(smem_u32(&aux->bar_o_ready[t]), 128);
            mbar_init(smem_u32(&aux->bar_pv_done[t]), 1);
            mbar_init(smem_u32(&aux->bar_mb_full[t]), 128);
            mbar_init(smem_u32(&aux->bar_mb_empty[t]), 128);
            mbar_init(smem_u32(&aux->bar_epi[t]), 128);
        }
        mbar_init(smem_u32(&aux->bar_drain), 1);
        aux->abort_flag = 0;
        mbar_fence_init();
    }
    if (warp == T::MMA_WARP) {
        tmem_alloc(smem_u32(&aux->tmem_base), T::TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = aux->tmem_base;
    const WaitCtx wc{&aux->abort_flag, args.err_word, args.wait_limit_ns};

    if (wg < T::NQ) {
        setmaxnreg_inc<T::REG_SOFTMAX>();
        prefill_softmax_role<T, CAUSAL>(wg, args, w, aux, tmem, wc);
    } else if (wg == T::CORR_WG) {
        setmaxnreg_dec<T::REG_CORR>();
        prefill_correction_role<T>(&tm_o, args, w, aux, tmem, sQ, wc);
    } else {
        setmaxnreg_dec<T::REG_OTHER>();
        if (warp == T::MMA_WARP)
            prefill_mma_role<T>(args, w, aux, tmem, sQ, sRing, wc);
        else if (warp == T::LOAD_WARP)
            prefill_load_role<T>(&tm_q, &tm_k, &tm_v, args, w, aux, sQ, sRing, wc);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == T::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, T::TMEM_COLS);
    }
}

// Host-side launch of one head-dimension instantiation.
template <int D>
cudaError_t launch_prefill_impl(const PrefillLaunch& p, cudaStream_t stream) {
    using T = PrefillTraits<D>;
    void (*kern)(CUtensorMap, CUtensorMap, CUtensorMap, CUtensorMap, PrefillArgs) =
        p.causal ? prefill_kernel<D, true> : prefill_kernel<D, false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         T::SMEM_TOTAL);
    if (e != cudaSuccess) return e;
    const dim3 grid((unsigned)p.args.num_mblk, (unsigned)p.args.Hq, (unsigned)p.args.B);
    kern<<<grid, T::THREADS, T::SMEM_TOTAL, stream>>>(p.tm_q, p.tm_k, p.tm_v, p.tm_o, p.args);
    return cudaGetLastError();
}

}  // namespace fa
