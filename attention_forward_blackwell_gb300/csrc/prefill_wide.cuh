// Prefill with 256-key score blocks (head_dim 96 and 128): one persistent
// CTA per SM, one Q tile of 128 rows per unit.  Dense launches without a
// window, paged caches or packed sequences run it, causal or not (causal
// units come heaviest first, as in the other kernels); the others run the
// two-tile kernels of prefill.cuh.
//
// Included by prefill.cuh after the roles and helpers it shares (the work
// split, the staged O drain, the final normaliser).
//
// GQA head packing (PACK instances, PrefillArgs::pack = P > 1): with short
// queries the 128 tile rows hold P query heads of one kv group x 128 / P
// positions ("b200-flash-attention4-planner" E.7: explicit head mapping and
// reuse), so that one stream of K/V tiles serves all P heads instead of a
// tile whose rows are mostly empty.  The Q map's box is {64, 128 / P, P}
// (the P heads' rows land in shared memory head after head, exactly the
// unpacked tile's layout), the O map's box {32, 16, 2} when a head has 16
// rows; the causal mask, the sink and the LSE take each row's own head and
// position (wide_row).  Measured on GB300 (B=64 Hq=32 Hkv=4, 16 queries
// over 4,096 keys): 93 -> 335 TFLOPS causal, 192 -> 671 non-causal.
//
// Why: from one issuing thread a tcgen05.mma of M = 128, K = 16 occupies
// the tensor pipe ~80 cycles for any N up to 128 and 128 cycles at N = 256
// (measured on GB300), so only N = 256 runs at the pipe's full rate.  The
// two-tile kernels issue score MMAs of N = 128 (the 128-key block), and
// their P lives in the upper half of the tile's score buffer, so a tile's
// next score MMA also waits for its value MMA.  Here a key block is 256
// keys: the score MMA S = Q K^T is one N = 256 instruction per K-step of 16
// head dims (half the score instructions per key, each at the full rate),
// and tensor memory holds S (256 columns), P (128 columns of bf16 pairs) and
// O (d columns) side by side, so that S(J+1) is issued as soon as the
// softmax has read S(J) into registers and runs while the softmax computes
// P(J) (the FlashAttention-4 planner's overlap of the score MMA of the next
// tile with the softmax of this one, "b200-flash-attention4-planner" A1,
// E.3).  The softmax computes P(J) into registers while PV(J-1) still reads
// the one P buffer and stores it once PV(J-1) has completed.  Measured on
// GB300 against the two-tile kernel: +4 % at 8,192 keys, +8 % at 4,096 keys
// (head_dim 128), +5 % at head_dim 96; a block takes ~3,050 cycles, bound by
// the softmax (both warpgroups work on the same block at the same time, where
// the two-tile kernel's softmaxes alternate).
//
// Roles (512 threads):
//   warps 0-7   softmax: warpgroup h takes the keys [128 h, 128 h + 128) of
//               each block for all 128 rows (thread = row = TMEM lane); the
//               two halves of a row exchange their block maxima through
//               shared memory, then share one running max (the O basis);
//   warps 8-11  correction: follows the running max from the same block
//               maxima, rebases O when it moved (lazily, as in the other
//               kernels), and at a unit's end drains O / l
//               to global memory through 2 KB staging buffers and TMA
//               stores while the next unit's first scores run;
//   warp 12     MMA issue (one lane): S(J+1), then PV(J);
//   warp 13     TMA producer: K as one 64-column chunk of 256 rows per ring
//               slot, V as two slots of 128 keys x all columns, in the order
//               the MMA lane consumes them.
//
// Scheduling, barrier phases and unit boundaries follow the persistent
// head_dim-256 kernel: unit i of CTA x is persist_unit(i, x, G); ring
// positions, key-block indices J and unit counts kq run on over the CTA's
// units, so every parity is a running one.
//
// Barrier protocol (every wait bounded):
//   s_full       S(J) complete (MMA commit), one phase per block;
//   xm[J & 1]    both halves' block maxima of block J posted (8 warps),
//                after each warp has read S(J) into registers: the softmax
//                halves take the other half's max from it, the MMA lane
//                issues S(J+1) into the score buffer after it, and the
//                correction warpgroup derives the rebase factor of block J
//                from the two maxima with the softmax's own operations (so
//                no mailbox carries it);
//   p_ready[J&1] P(J) written (8 softmax warps) and O rebased (4 correction
//                warps); PV(J) waits for it;
//   pv_done[J&1] PV(J) complete; P(J+1) is written only after it;
//   fin          a unit's row statistics posted (8 warps);
//   qfree        the unit's last score MMA complete (the producer then loads
//                the next unit's Q);
//   odrained     the unit's O read out of tensor memory (4 correction
//                warps); the next unit's first PV and final statistics wait
//                for it.
// A copy indexed by J & 1 is never two phases ahead of a reader: the
// halves post block J+2's maxima after S(J+2) completed, which the MMA lane
// issued after PV(J), which waited for P-ready(J), which includes the
// correction's arrival for block J (made after it read block J's maxima);
// the halves read the other's block-J max before they arrive for block
// J+1, which the MMA lane waits for before S(J+2).  (Measured on GB300: the
// rebase factor computed by the correction warpgroup instead of posted by
// one softmax warpgroup, and no separate barrier for the score buffer, are
// +2 to +4 %.)
#pragma once

namespace fa {

constexpr int kWideSlots = 5;   // ring slots of the 256-key kernel

template <int D, bool C = false, bool PK = false, bool SP = false>
struct WideTraits {
    static constexpr bool CAUSAL = C;               // causal mask (bottom-right aligned)
    static constexpr bool PACK = PK;                // GQA head packing (PrefillArgs::pack > 1)
    static constexpr bool SPLIT = SP;               // units split along the keys, one piece per CTA
    static constexpr int BM = 128;                  // query rows of a unit = TMEM lanes
    static constexpr int BN = 256;                  // keys per score block
    static constexpr int NQ = 1;                    // (shared work split: one Q tile)
    static constexpr int DV_SPLIT = 1;
    static constexpr int D_COLS = D;
    static constexpr bool BOX4 = false;             // 3-D copies of one chunk each
    static constexpr int NCH = (D + 63) / 64;       // 64-column chunks of a row
    static constexpr int CHUNK = 128 * 128;         // one chunk of 128 rows, bytes
    static constexpr int QTILE = NCH * CHUNK;
    static constexpr int KSTEPS = D / 16;           // score MMA steps of K = 16
    static constexpr int SLOT = 32768;              // ring slot, bytes
    static constexpr int KP = NCH;                  // slots of a K block: one chunk of 256 rows each
    static constexpr int VP = 2;                    // slots of a V block: 128 keys x NCH chunks each
    static constexpr int VKEYS = BN / VP;
    static constexpr int NSLOT = kWideSlots;
    static constexpr int THREADS = 512;
    static constexpr int CORR_WG = 2;
    static constexpr int MMA_WARP = 12;
    static constexpr int LOAD_WARP = 13;
    static constexpr uint32_t TMEM_COLS = 512;
    static constexpr uint32_t S_COL = 0;            // S: 256 fp32 columns
    static constexpr uint32_t P_COL = 256;          // P: 256 keys as 128 columns of bf16 pairs
    static constexpr uint32_t O_COL = 384;          // O: d fp32 columns
    static constexpr int STAGE_BUFS = 3;            // O staging: 3 x 2 KB per correction warp
    static constexpr int SMEM_Q = QTILE;
    static constexpr int SMEM_RING = NSLOT * SLOT;
    static constexpr int SMEM_AUX = 8192;
    static constexpr int SMEM_STAGE = 4 * STAGE_BUFS * 2048;
    static constexpr int SMEM_TOTAL = 1024 + SMEM_Q + SMEM_RING + SMEM_AUX + SMEM_STAGE;
    // register split of the 512 x 128 launch allocation: the two softmax
    // warpgroups, the correction warpgroup, the MMA / producer warpgroup
    static constexpr uint32_t LAUNCH_REGS = 128;
    // (measured on GB300: 176 / 88 / 72 and 176 / 96 / 64 are 4-6 % slower:
    // the MMA-issue and producer warps need their 80)
    struct Regs {
        static constexpr uint32_t SOFTMAX = 168;
        static constexpr uint32_t CORR = 96;
        static constexpr uint32_t OTHER = 80;
        static_assert(SOFTMAX > LAUNCH_REGS && CORR < LAUNCH_REGS && OTHER < LAUNCH_REGS,
                      "setmaxnreg targets must move away from the launch allocation");
        static_assert(8 * 32 * SOFTMAX + 4 * 32 * CORR + 4 * 32 * OTHER <= THREADS * LAUNCH_REGS,
                      "register split exceeds the launch allocation");
    };
    static_assert(D == 96 || D == 128, "256-key blocks: head_dim 96 or 128");
    static_assert(NCH == 2 && SLOT == 256 * 128 && SLOT == NCH * CHUNK && KSTEPS * 16 == D,
                  "a K slot is one chunk of 256 rows, a V slot 128 keys of both chunks");
    static_assert(O_COL + D <= TMEM_COLS, "S, P and O must fit the tensor memory");
    static_assert(SMEM_TOTAL <= 232448, "shared memory per CTA exceeds the sm_103 limit");
};

struct WideAux {
    uint64_t bar_q;
    uint64_t bar_full[kWideSlots];
    uint64_t bar_empty[kWideSlots];
    uint64_t bar_s_full;
    uint64_t bar_xm[2];
    uint64_t bar_p_ready[2];
    uint64_t bar_pv_done[2];
    uint64_t bar_fin;
    uint64_t bar_qfree;
    uint64_t bar_odrained;
    uint64_t bar_tail;
    uint64_t bar_drain;
    uint64_t bar_split_a;     // a piece's partial result written (4 correction warps)
    uint32_t tmem_base;
    int abort_flag;
    int merge_last;           // this CTA's piece arrived last: it merges the unit
    int merge_unit[4];        // tail, head, batch entry, first row of that unit
    float xm[2][2][128];      // [J & 1][half][row] block maxima
    float mb_l[2][128];       // [half][row] row sums of the unit
};

// Work items of a launch: whole units only (n_full), or (SPLIT instances)
// pieces as well.  The bound is n_full unless the instance splits, so that
// the compiler sees every item as a whole unit and drops prefill_work's piece
// arithmetic from the roles (measured on GB300: bounding the unsplit
// kernels' loops by n_work instead, the same value at run time, made them
// 10 % slower).
template <class T>
__device__ __forceinline__ int wide_items(const PrefillArgs& a) {
    return T::SPLIT ? a.n_work : a.n_full;
}

// Unit u of the 256-key kernel.  Without packing, prefill_work's unit
// (batch entry, query head, block of 128 query rows).  With P = a.pack heads
// per tile: (batch entry, heads h .. h + P - 1 of one kv group, block of
// R = 128 / P query positions), ordered as prefill_work orders its units
// (causal: query block slowest, heaviest first); row0 is the block's first
// position, and the key blocks are those its last position sees.
template <class T>
__device__ __forceinline__ PrefillWork wide_work(const PrefillArgs& a, int u) {
    if constexpr (!T::PACK) {
        return prefill_work<T, T::CAUSAL, false, false>(a, u);
    } else {
        PrefillWork w;
        int kb = 0, ke = 0x7fffffff;   // key blocks [kb, ke) of a piece
        w.piece = -1;
        w.tail = -1;
        if (u >= a.n_full) {   // piece k of split unit `tail`, as prefill_work cuts them
            const int q = u - a.n_full;
            const int k = q % a.split;
            w.tail = q / a.split;
            w.piece = q;
            kb = (int)((long long)k * a.nk / a.split);
            ke = (int)((long long)(k + 1) * a.nk / a.split);
            u = a.n_full + w.tail;
        }
        const int rows = T::BM / a.pack;            // query positions per head
        const int ng = a.Hq / a.pack;               // head groups per batch entry
        const int nbh = a.B * ng;
        const int x = T::CAUSAL ? u / nbh : u % a.num_mblk;
        const int hb = T::CAUSAL ? u % nbh : u / a.num_mblk;
        const int mblk = T::CAUSAL ? (a.num_mblk - 1 - x) : x;
        w.b = hb / ng;
        w.h = (hb % ng) * a.pack;
        w.hk = w.h / a.group;
        int L = a.Sk;
        if (a.seqlens_k != nullptr) L = max(0, min(a.seqlens_k[w.b], a.Sk));
        w.L = L;
        w.off = L - a.Sq;
        w.row0 = mblk * rows;
        int last = L - 1;   // last key any row of the tile can see
        if (T::CAUSAL) last = min(last, w.row0 + rows - 1 + w.off);
        const int n = last >= 0 ? last / T::BN + 1 : 0;
        const int cnt = min(n, ke) - kb;
        w.kb = kb;
        w.n_kv[0] = w.n_kv[1] = cnt > 0 ? cnt : 0;
        w.n_max = w.n_kv[0];
        w.Lq = w.q0 = w.k0 = 0;
        w.dv0 = 0;
        return w;
    }
}

// Query head and position of tile row r of unit w.
template <class T>
__device__ __forceinline__ void wide_row(const PrefillArgs& a, const PrefillWork& w, int r,
                                         int& h, int& pos) {
    if constexpr (T::PACK) {
        const int rows = T::BM / a.pack;
        h = w.h + r / rows;
        pos = w.row0 + r % rows;
    } else {
        h = w.h;
        pos = w.row0 + r;
    }
}

// L2 prefetch of unit u's Q tile (the Q map's box: 128 rows of one head, or
// R rows x P heads).
template <class T>
__device__ __forceinline__ void wide_prefetch_q(const CUtensorMap* tm_q, const PrefillArgs& a,
                                                int u) {
    if constexpr (!T::PACK) {
        prefetch_q_of<T, T::CAUSAL, false, false>(tm_q, a, u);
    } else {
        const PrefillWork w2 = wide_work<T>(a, u);
        if (w2.n_max <= 0) return;
#pragma unroll
        for (int c = 0; c < T::NCH; ++c)
            tma_prefetch_l2_3d(tm_q, c * 64, w2.row0, w2.b * a.Hq + w2.h);
    }
}

// A unit without keys: O = 0 and LSE = log of the sink term (or -inf), by
// the correction warpgroup (thread = row).
template <class T>
__device__ void wide_write_empty(const PrefillArgs& a, const PrefillWork& w) {
    if constexpr (!T::PACK) {
        write_empty_unit<T>(a, w);
    } else {
        const int r = ((threadIdx.x >> 5) & 3) * 32 + (threadIdx.x & 31);
        int h, pos;
        wide_row<T>(a, w, r, h, pos);
        float lf, mf;
        const float inv_l = final_scale(a, h, 0.f, -INFINITY, lf, mf);
        uint16_t* orow = a.o + (((size_t)w.b * a.Hq + h) * a.Sq + pos) * T::D_COLS;
        store_o_rows_direct<T>(0u, 0u, orow, pos < a.Sq, 0, inv_l, 0, T::D_COLS / 32);
        if (pos < a.Sq)
            a.lse[((size_t)w.b * a.Hq + h) * a.Sq + pos] =
                (lf > 0.f) ? (mf + lg2_approx(lf)) * kLn2 : -INFINITY;
    }
}

// Zeroes rows [r0, 128) of both 64-column chunks of a V slot (all 32 lanes
// of the calling warp), then makes the writes visible to the tensor core.
template <class T>
__device__ __forceinline__ void wide_zero_value_rows(uint32_t slot_addr, int r0) {
    const int lane = threadIdx.x & 31;
    const int granules = (T::VKEYS - r0) * 8;   // 16-byte granules per chunk
#pragma unroll
    for (int c = 0; c < T::NCH; ++c) {
        const uint32_t base = slot_addr + c * T::CHUNK + r0 * 128;
        for (int g = lane; g < granules; g += 32)
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(base + g * 16), "r"(0)
                         : "memory");
    }
    fence_proxy_async_smem();
    __syncwarp();
}

// Producer over the CTA's units: per unit K_0, the unit's Q (once the
// previous unit's last score MMA has completed), then K_{j+1} and V_j for
// every block j (the MMA lane's order).  K: one 3-D copy of a {64, 256} box per chunk (tm_k);
// V: two 3-D copies of {64, 128} boxes per half (tm_v); V rows past the
// sequence's last key are zeroed before the slot is published (a zero
// probability times a non-finite value would poison O).
template <class T>
__device__ void wide_load_role(const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                               const CUtensorMap* tm_v, const PrefillArgs& a, WideAux* aux,
                               uint32_t sQ, uint32_t sRing, const WaitCtx& wc) {
    const int lane = threadIdx.x & 31;
    const int G = (int)gridDim.x, x = (int)blockIdx.x;
    const uint32_t bar_q = smem_u32(&aux->bar_q);
    if (lane == 0) {
        tma_prefetch_desc(tm_q);
        tma_prefetch_desc(tm_k);
        tma_prefetch_desc(tm_v);
    }
    int p = 0, ntail = 0, kq = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
        const int u = persist_unit(i, x, G);
        if (u >= wide_items<T>(a)) break;
        const PrefillWork w = wide_work<T>(a, u);
        if (w.n_max <= 0) continue;
        const int plane = w.b * a.Hkv + w.hk;
        // next ring position's slot, once its previous contents were consumed
        auto acquire = [&](uint32_t& dst, uint32_t& full) -> bool {
            const uint32_t slot = ring_slot<T>(p);
            if (!mbar_wait(smem_u32(&aux->bar_empty[slot]), ring_phase<T>(p) ^ 1u, wc,
                           kErrWaitTimeout | kSiteLoadEmpty))
                return false;
            dst = sRing + slot * T::SLOT;
            full = smem_u32(&aux->bar_full[slot]);
            return true;
        };
        auto load_k = [&](int j, int c) -> bool {
            uint32_t dst, full;
            if (!acquire(dst, full)) return false;
            if (lane == 0) {
                mbar_arrive_expect_tx(full, (uint32_t)T::SLOT);
                tma_load_3d(dst, tm_k, c * 64, (w.kb + j) * T::BN, plane, full);
            }
            __syncwarp();
            ++p;
            return true;
        };
        auto load_v = [&](int j, int hh) -> bool {
            uint32_t dst, full;
            if (!acquire(dst, full)) return false;
            const int r0 = (w.kb + j) * T::BN + hh * T::VKEYS;   // first key of the slot
            const int rv = w.L - r0;                              // valid keys in it
            if (rv < T::VKEYS) {
                const uint32_t tail = smem_u32(&aux->bar_tail);
                if (lane == 0) {
                    mbar_arrive_expect_tx(tail, (uint32_t)T::SLOT);
                    load_chunks<T, T::NCH>(dst, tm_v, 0, r0, plane, tail);
                }
                if (!mbar_wait(tail, (uint32_t)(ntail & 1), wc, kErrWaitTimeout | kSiteLoadTail))
                    return false;
                ++ntail;
                wide_zero_value_rows<T>(dst, rv > 0 ? rv : 0);
                if (lane == 0) mbar_arrive(full);
            } else if (lane == 0) {
                mbar_arrive_expect_tx(full, (uint32_t)T::SLOT);
                load_chunks<T, T::NCH>(dst, tm_v, 0, r0, plane, full);
            }
            __syncwarp();
            ++p;
            return true;
        };
        // K_0 first: its slots are free while the previous unit's last
        // score MMA still reads Q
        for (int c = 0; c < T::KP && ok; ++c) ok = load_k(0, c);
        if (!ok) break;
        if (kq > 0 && !mbar_wait(smem_u32(&aux->bar_qfree), (uint32_t)((kq - 1) & 1), wc,
                                 kErrWaitTimeout | kSiteLoadQfree))
            break;
        if (lane == 0) {
            mbar_arrive_expect_tx(bar_q, (uint32_t)T::QTILE);
            load_chunks<T, T::NCH>(sQ, tm_q, 0, w.row0, w.b * a.Hq + w.h, bar_q);
            const int un = persist_unit(i + 1, x, G);   // this CTA's next unit
            if (un < wide_items<T>(a)) wide_prefetch_q<T>(tm_q, a, un);
        }
        __syncwarp();
        ++kq;
        for (int j = 0; j < w.n_max && ok; ++j) {
            if (j + 1 < w.n_max)
                for (int c = 0; c < T::KP && ok; ++c) ok = load_k(j + 1, c);
            for (int hh = 0; hh < T::VP && ok; ++hh) ok = load_v(j, hh);
        }
    }
    // every copy issued must have landed before the CTA exits
    if (lane == 0) {
        if (kq > 0) mbar_wait_drain(bar_q, (uint32_t)((kq - 1) & 1), a.wait_limit_ns);
        for (int q = p > T::NSLOT ? p - T::NSLOT : 0; q < p; ++q)
            mbar_wait_drain(smem_u32(&aux->bar_full[ring_slot<T>(q)]), ring_phase<T>(q),
                            a.wait_limit_ns);
    }
    __syncwarp();
}

// MMA issue over the CTA's units (one lane).  Block J: S(J+1) once the
// softmax has read S(J) out of the buffer (both halves posted their block
// maxima) and K_{j+1} has landed, then PV(J) once P(J) is ready.  Each ring
// slot is released by a commit after the MMAs that read it.
template <class T>
__device__ void wide_mma_role(const PrefillArgs& a, WideAux* aux, uint32_t tmem, uint32_t sQ,
                              uint32_t sRing, const WaitCtx& wc, unsigned long long* tr) {
    const int lane = threadIdx.x & 31;
    if (lane != 0) {
        __syncwarp();
        return;
    }
    const int G = (int)gridDim.x, x = (int)blockIdx.x;
    const uint32_t qd0 = sdesc_lo_sw128(sQ, 16);             // K-major Q
    const uint32_t kd0 = sdesc_lo_sw128(sRing, 16);          // K-major K, 256 rows
    const uint32_t vd0 = sdesc_lo_sw128(sRing, T::CHUNK);    // MN-major V, chunks 16 KB apart
    constexpr uint32_t idesc_s = idesc_bf16_f32(128, T::BN, false, false);
    constexpr uint32_t idesc_v = idesc_bf16_f32(128, T::D_COLS, false, true);
    int p = 0;   // ring position of the next slot (the producer's order)
    auto next_slot = [&](unsigned site) -> bool {
        if (!mbar_wait_lane(smem_u32(&aux->bar_full[ring_slot<T>(p)]), ring_phase<T>(p), wc,
                            kErrWaitTimeout | site))
            return false;
        tc_fence_after();
        return true;
    };
    auto slot_desc = [&](uint32_t d0) { return d0 + (uint32_t)((ring_slot<T>(p) * T::SLOT) >> 4); };
    // S(J) = Q K_j^T over 256 keys: one N = 256 instruction per K-step
    auto score = [&](int J) -> bool {
        trace_mark(tr, kTrMma, J, 0);
        if (J > 0) {   // the softmax has read S(J-1) out of the buffer
            if (!mbar_wait_lane(smem_u32(&aux->bar_xm[(J - 1) & 1]), (uint32_t)(((J - 1) >> 1) & 1),
                                wc, kErrWaitTimeout | kSiteMmaSfree))
                return false;
            tc_fence_after();
        }
        trace_mark(tr, kTrMma, J, 1);
        for (int c = 0; c < T::KP; ++c) {
            if (!next_slot(kSiteMmaK)) return false;
            trace_mark(tr, kTrMma, J, 2 + c);
            const uint32_t kd = slot_desc(kd0);
#pragma unroll
            for (int kin = 0; kin < 4; ++kin) {
                const int kk = c * 4 + kin;
                if (kk < T::KSTEPS)
                    umma_ss_lo(tmem + T::S_COL, qd0 + kstep_off(kk), kd + (uint32_t)((kin * 32) >> 4),
                               idesc_s, kk > 0 ? 1u : 0u);
            }
            tc_commit(smem_u32(&aux->bar_empty[ring_slot<T>(p)]));
            ++p;
        }
        tc_commit(smem_u32(&aux->bar_s_full));
        trace_mark(tr, kTrMma, J, 4);
        return true;
    };
    int J0 = 0, kq = 0;
    bool ok = true;
    for (int i = 0; ok; ++i) {
        const int u = persist_unit(i, x, G);
        if (u >= wide_items<T>(a)) break;
        const PrefillWork w = wide_work<T>(a, u);
        const int n = w.n_max;
        if (n <= 0) continue;
        if (!mbar_wait_lane(smem_u32(&aux->bar_q), (uint32_t)(kq & 1), wc,
                            kErrWaitTimeout | kSiteMmaQ))
            break;
        tc_fence_after();
        if (!score(J0)) break;
        if (n == 1) tc_commit(smem_u32(&aux->bar_qfree));   // Q no longer read
        for (int j = 0; j < n && ok; ++j) {
            const int J = J0 + j;
            if (j + 1 < n) {
                if (!score(J + 1)) {
                    ok = false;
                    break;
                }
                if (j + 2 == n) tc_commit(smem_u32(&aux->bar_qfree));   // Q no longer read
            }
            if (!mbar_wait_lane(smem_u32(&aux->bar_p_ready[J & 1]), (uint32_t)((J >> 1) & 1), wc,
                                kErrWaitTimeout | kSiteMmaP)) {
                ok = false;
                break;
            }
            trace_mark(tr, kTrMma, J, 5);
            tc_fence_after();
            // the unit's first value MMA overwrites O: the previous unit's O
            // must have been read out
            if (j == 0 && kq > 0) {
                if (!mbar_wait_lane(smem_u32(&aux->bar_odrained), (uint32_t)((kq - 1) & 1), wc,
                                    kErrWaitTimeout | kSiteMmaOdrained)) {
                    ok = false;
                    break;
                }
                tc_fence_after();
            }
            for (int hh = 0; hh < T::VP; ++hh) {
                if (!next_slot(kSiteMmaV)) {
                    ok = false;
                    break;
                }
                trace_mark(tr, kTrMma, J, 6 + hh);
                const uint32_t vd = slot_desc(vd0);
#pragma unroll
                for (int kk = 0; kk < T::VKEYS / 16; ++kk)
                    umma_ts_lo(tmem + T::O_COL, tmem + T::P_COL + (uint32_t)((hh * (T::VKEYS / 16) + kk) * 8),
                               vd + (uint32_t)((kk * 2048) >> 4), idesc_v,
                               (j > 0 || hh > 0 || kk > 0) ? 1u : 0u);
                tc_commit(smem_u32(&aux->bar_empty[ring_slot<T>(p)]));
                ++p;
            }
            if (ok) tc_commit(smem_u32(&aux->bar_pv_done[J & 1]));
            trace_mark(tr, kTrMma, J, 8);
        }
        J0 += n;
        ++kq;
    }
    // every MMA issued must have completed before tensor memory is freed
    {
        const uint32_t drain = smem_u32(&aux->bar_drain);
        tc_commit(drain);
        mbar_wait_drain(drain, 0, a.wait_limit_ns);
    }
    __syncwarp();
}

// Softmax of one unit by warpgroup h (keys [128 h, 128 h + 128) of every
// block; thread = row).  Per block: read the 128 scores, post the block max
// of the half (which also releases the score buffer) and take the other
// half's, move the running max lazily (the same rule as the other kernels;
// the correction warpgroup follows it from the same maxima), compute
// P = exp2(s scale log2e - m) as bf16 and the half's row sum, and store P
// once PV(J-1) has read the P buffer.  At the unit's end the two halves'
// row sums are posted for the epilogue.  Returns false if a wait gave up.
template <class T>
__device__ bool wide_softmax_unit(int h, const PrefillArgs& a, const PrefillWork& w,
                                  WideAux* aux, uint32_t tmem, const WaitCtx& wc, int J0, int kq,
                                  unsigned long long* tr) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if ((warp & 3) != 0 || lane != 0) tr = nullptr;
    const int trole = h == 0 ? kTrSoftmax0 : kTrSoftmax1;
    const int r = (warp & 3) * 32 + lane;                    // row = TMEM lane
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    int lim = w.L - 1;   // last visible key of this row
    if (T::CAUSAL) {
        int hr, pos;
        wide_row<T>(a, w, r, hr, pos);
        lim = min(lim, pos + w.off);
    }
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY;   // running max of scaled scores, log2 units (the basis)
    float l_run = 0.f;         // this half's running row sum in that basis
    for (int j = 0; j < w.n_max; ++j) {
        const int J = J0 + j;
        const int sb = J & 1;
        const uint32_t par = (uint32_t)((J >> 1) & 1);
        uint32_t u[4][32];
        if (!mbar_wait(smem_u32(&aux->bar_s_full), (uint32_t)(J & 1), wc,
                       kErrWaitTimeout | kSiteSmS))
            return false;
        trace_mark(tr, trole, J, 0);
        tc_fence_after();
        // the half's 128 scores in two 64-column loads (measured +1 % at
        // head_dim 96 against four 32-column ones; one 128-column load needs
        // more registers than the launch allocation)
        tmem_ld64(lane_base + T::S_COL + h * 128, *reinterpret_cast<uint32_t(*)[2][32]>(&u[0][0]));
        tmem_ld64(lane_base + T::S_COL + h * 128 + 64,
                  *reinterpret_cast<uint32_t(*)[2][32]>(&u[2][0]));
        tmem_wait_ld();
        trace_mark(tr, trole, J, 1);
        float s[128];
#pragma unroll
        for (int c = 0; c < 128; ++c) s[c] = __uint_as_float(u[c >> 5][c & 31]);
        const int kv0 = (w.kb + j) * T::BN + h * 128;   // first key of the half
        if (lim - kv0 < 127) {
            const int nvis = lim - kv0 + 1;
#pragma unroll
            for (int c = 0; c < 128; ++c) s[c] = (c < nvis) ? s[c] : -INFINITY;
        }
        float mq[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            float m = fmax3(s[32 * q], s[32 * q + 1], s[32 * q + 2]);
#pragma unroll
            for (int c = 3; c < 31; c += 2) m = fmax3(m, s[32 * q + c], s[32 * q + c + 1]);
            mq[q] = fmaxf(m, s[32 * q + 31]);
        }
        const float mx_h = fmaxf(fmax3(mq[0], mq[1], mq[2]), mq[3]);
        trace_mark(tr, trole, J, 5);
        aux->xm[sb][h][r] = mx_h;
        tc_fence_before();   // (this arrival also releases the score buffer to S(J+1))
        mbar_arrive_warp(smem_u32(&aux->bar_xm[sb]));
        if (!mbar_wait(smem_u32(&aux->bar_xm[sb]), par, wc, kErrWaitTimeout | kSiteSmXm))
            return false;
        trace_mark(tr, trole, J, 2);
        // the row's block max, and the lazy move of the basis (as in the
        // other kernels); both halves compute the same values
        const float m_new = fmaxf(m_run, fmaxf(mx_h, aux->xm[sb][h ^ 1][r]) * sl2);
        float alpha = 1.f;
        if (m_new > m_run + kRescaleThreshold) {
            alpha = ex2_approx(m_run - m_new);   // 0 when m_run = -inf
            m_run = m_new;
        }
        // P(J) is computed into registers while PV(J-1) still reads P(J-1)
        // out of the one P buffer; only its stores wait for PV(J-1) (and
        // storing the first half before computing the second keeps the
        // registers within the softmax's share without spills: measured
        // +0.5 % against storing both halves at the end)
        const float base = (m_run == -INFINITY) ? 0.f : m_run;
        const float2 sl2x2 = make_float2(sl2, sl2);
        const float2 nbase = make_float2(-base, -base);
        float2 rs[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                        make_float2(0.f, 0.f)};
        uint32_t pk[2][32];
        const uint32_t pcol = lane_base + T::P_COL + h * 64;
        // the first 64 keys' P, then (once PV(J-1) has completed: P(J)
        // overwrites P(J-1)) their store while the other 64 are computed
#pragma unroll
        for (int c = 0; c < 64; ++c) {
            const float2 xv = ffma2(make_float2(s[2 * c], s[2 * c + 1]), sl2x2, nbase);
            const float2 pv = make_float2(ex2_approx(xv.x), ex2_approx(xv.y));
            rs[c & 3] = fadd2(rs[c & 3], pv);
            pk[c >> 5][c & 31] = pack_bf16x2(pv.x, pv.y);
            if (c == 31) {
                trace_mark(tr, trole, J, 3);
                if (J > 0) {
                    if (!mbar_wait(smem_u32(&aux->bar_pv_done[(J - 1) & 1]),
                                   (uint32_t)(((J - 1) >> 1) & 1), wc,
                                   kErrWaitTimeout | kSiteSmPv))
                        return false;
                    tc_fence_after();
                }
                trace_mark(tr, trole, J, 6);
                tmem_st32(pcol, pk[0]);
            }
        }
        const float2 rs01 = fadd2(rs[0], rs[1]), rs23 = fadd2(rs[2], rs[3]);
        const float2 rsum = fadd2(rs01, rs23);
        l_run = fmaf(l_run, alpha, rsum.x + rsum.y);
        tmem_st32(pcol + 32, pk[1]);
        tmem_wait_st();
        tc_fence_before();
        mbar_arrive_warp(smem_u32(&aux->bar_p_ready[sb]));
        trace_mark(tr, trole, J, 4);
    }
    // the previous unit's statistics must have been read (the correction
    // warpgroup arrives on O-drained after reading them)
    if (kq > 0 && !mbar_wait(smem_u32(&aux->bar_odrained), (uint32_t)((kq - 1) & 1), wc,
                             kErrWaitTimeout | kSiteSmOdrained))
        return false;
    aux->mb_l[h][r] = l_run;
    mbar_arrive_warp(smem_u32(&aux->bar_fin));
    return true;
}

// Correction of one unit (warpgroup CORR_WG, thread = row): follows the
// running max from the halves' block maxima, rebases O before PV(J) when it
// moved, then drains O / l (bf16) through
// the warp's staging buffers and TMA stores (tm_o32: box {32, 32, 1}),
// stores LSE = ln2 (m + log2 l) and arrives on O-drained.
template <class T>
__device__ bool wide_correction_unit(const CUtensorMap* tm_o32, const PrefillArgs& a,
                                     const PrefillWork& w, WideAux* aux, uint32_t tmem,
                                     uint32_t sQ, const WaitCtx& wc, int J0, int kq) {
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int r = (warp & 3) * 32 + lane;
    const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const int n = w.n_max;
    const float sl2 = a.scale_log2;
    float m_run = -INFINITY;   // the softmax's running max, by the same operations
    for (int j = 0; j < n; ++j) {
        const int J = J0 + j;
        const int sb = J & 1;
        // the halves' block maxima of block J, and the rebase factor the
        // softmax derives from them
        if (!mbar_wait(smem_u32(&aux->bar_xm[sb]), (uint32_t)((J >> 1) & 1), wc,
                       kErrWaitTimeout | kSiteCorrMbox))
            return false;
        const float m_new = fmaxf(m_run, fmaxf(aux->xm[sb][0][r], aux->xm[sb][1][r]) * sl2);
        float alpha = 1.f;
        if (m_new > m_run + kRescaleThreshold) {
            alpha = ex2_approx(m_run - m_new);   // 0 when m_run = -inf
            m_run = m_new;
        }
        if (j > 0 && __any_sync(0xffffffffu, alpha < 1.f)) {
            // O must hold PV(J-1) before it is rebased
            if (!mbar_wait(smem_u32(&aux->bar_pv_done[(J - 1) & 1]),
                           (uint32_t)(((J - 1) >> 1) & 1), wc, kErrWaitTimeout | kSiteCorrPv))
                return false;
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < T::D_COLS / 32; ++c) {
                uint32_t v[32];
                tmem_ld32(lane_base + T::O_COL + c * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int e = 0; e < 32; ++e) v[e] = __float_as_uint(__uint_as_float(v[e]) * alpha);
                tmem_st32(lane_base + T::O_COL + c * 32, v);
            }
            tmem_wait_st();
        }
        tc_fence_before();
        mbar_arrive_warp(smem_u32(&aux->bar_p_ready[sb]));   // O safe for PV(J)
    }
    if (!mbar_wait(smem_u32(&aux->bar_fin), (uint32_t)(kq & 1), wc, kErrWaitTimeout | kSiteEpiMbox))
        return false;
    const float l = aux->mb_l[0][r] + aux->mb_l[1][r];
    const float m = m_run;
    // O is final once PV(J0 + n - 1) completed (value MMAs into one
    // accumulator complete in issue order)
    const int Jl = J0 + n - 1;
    if (!mbar_wait(smem_u32(&aux->bar_pv_done[Jl & 1]), (uint32_t)((Jl >> 1) & 1), wc,
                   kErrWaitTimeout | kSiteEpiPv))
        return false;
    tc_fence_after();
    if constexpr (T::SPLIT) {
        if (w.piece >= 0) {
            // a piece of a split unit: unnormalised O (in the basis m), m
            // and l -> the piece's scratch slot; the last piece to arrive
            // merges the unit at the kernel's end
            float4* po = reinterpret_cast<float4*>(a.part_o +
                                                   (size_t)w.piece * (T::D_COLS * T::BM));
#pragma unroll 1
            for (int c32 = 0; c32 < T::D_COLS / 32; ++c32) {
                uint32_t v[32];
                tmem_ld32(lane_base + T::O_COL + c32 * 32, v);
                tmem_wait_ld();
#pragma unroll
                for (int q = 0; q < 8; ++q)
                    po[(size_t)(c32 * 8 + q) * T::BM + r] =
                        make_float4(__uint_as_float(v[4 * q]), __uint_as_float(v[4 * q + 1]),
                                    __uint_as_float(v[4 * q + 2]), __uint_as_float(v[4 * q + 3]));
            }
            float* ml = a.part_ml + (size_t)w.piece * 2 * T::BM;
            ml[r] = m;
            ml[T::BM + r] = l;
            tc_fence_before();
            mbar_arrive_warp(smem_u32(&aux->bar_odrained));
            split_arrive<T>(a, w, aux, wc);
            return true;
        }
    }
    float lf, mf;
    int h, row;   // this row's query head and position
    wide_row<T>(a, w, r, h, row);
    const float inv_l = final_scale(a, h, l, m, lf, mf);
    // the warp's first row: its 32 rows are one head's, or (16 positions per
    // head) two heads', which the O map's box covers
    int wh, wrow;
    wide_row<T>(a, w, (warp & 3) * 32, wh, wrow);
    uint16_t* obase = a.o + (((size_t)w.b * a.Hq + wh) * a.Sq + wrow) * T::D_COLS;
    store_o_rows_staged<T, 2>(lane_base, T::O_COL, obase, T::D_COLS, a.Sq - wrow, n, inv_l, 0,
                              T::D_COLS / 32, stage_of<T>(sQ, warp), tm_o32, 0, wrow,
                              w.b * a.Hq + wh);
    tc_fence_before();
    mbar_arrive_warp(smem_u32(&aux->bar_odrained));
    if (row < a.Sq)
        a.lse[((size_t)w.b * a.Hq + h) * a.Sq + row] =
            (lf > 0.f) ? (mf + lg2_approx(lf)) * kLn2 : -INFINITY;
    return true;
}

template <int D, bool CAUSAL, bool PACK, bool SPLIT>
__global__ void __launch_bounds__(WideTraits<D>::THREADS, 1)
    prefill_kernel_wide(const __grid_constant__ CUtensorMap tm_q,
                        const __grid_constant__ CUtensorMap tm_k,
                        const __grid_constant__ CUtensorMap tm_v,
                        const __grid_constant__ CUtensorMap tm_o32, const PrefillArgs args) {
    using T = WideTraits<D, CAUSAL, PACK, SPLIT>;
    static_assert(sizeof(WideAux) <= T::SMEM_AUX, "auxiliary shared block too large");
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    const uint32_t raw = smem_u32(smem_raw);
    const uint32_t sQ = (raw + 1023u) & ~1023u;   // 1024-aligned: swizzle atoms
    const uint32_t sRing = sQ + T::SMEM_Q;
    auto* aux = reinterpret_cast<WideAux*>(smem_raw + (sQ - raw) + T::SMEM_Q + T::SMEM_RING);
    const int warp = threadIdx.x >> 5;
    const int wg = warp >> 2;

    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&aux->bar_q), 1);
        for (int i = 0; i < T::NSLOT; ++i) {
            mbar_init(smem_u32(&aux->bar_full[i]), 1);
            mbar_init(smem_u32(&aux->bar_empty[i]), 1);
        }
        mbar_init(smem_u32(&aux->bar_s_full), 1);
        for (int i = 0; i < 2; ++i) {
            mbar_init(smem_u32(&aux->bar_xm[i]), 8);       // 8 softmax warps
            mbar_init(smem_u32(&aux->bar_p_ready[i]), 12); // 8 softmax + 4 correction warps
            mbar_init(smem_u32(&aux->bar_pv_done[i]), 1);
        }
        mbar_init(smem_u32(&aux->bar_fin), 8);
        mbar_init(smem_u32(&aux->bar_qfree), 1);
        mbar_init(smem_u32(&aux->bar_odrained), 4);        // 4 correction warps
        mbar_init(smem_u32(&aux->bar_tail), 1);
        mbar_init(smem_u32(&aux->bar_drain), 1);
        mbar_init(smem_u32(&aux->bar_split_a), 4);         // 4 correction warps
        aux->abort_flag = 0;
        aux->merge_last = 0;
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
    const WaitCtx wc{smem_u32(&aux->abort_flag), (uint32_t)args.wait_limit_ns, args.err_word};
    const int G = (int)gridDim.x, x = (int)blockIdx.x;
    unsigned long long* tr =
        (FA_PREFILL_TRACE && args.trace != nullptr && x == args.trace_block) ? args.trace : nullptr;

    if (wg < 2) {
        setmaxnreg_inc<T::Regs::SOFTMAX>();
        int J0 = 0, kq = 0;
        for (int i = 0;; ++i) {
            const int u = persist_unit(i, x, G);
            if (u >= wide_items<T>(args) || ld_volatile_shared(wc.abort_flag) != 0) break;
            const PrefillWork w = wide_work<T>(args, u);
            if (w.n_max <= 0) continue;
            if (!wide_softmax_unit<T>(wg, args, w, aux, tmem, wc, J0, kq, tr)) break;
            J0 += w.n_max;
            ++kq;
        }
    } else if (wg == T::CORR_WG) {
        setmaxnreg_dec<T::Regs::CORR>();
        int J0 = 0, kq = 0;
        for (int i = 0;; ++i) {
            const int u = persist_unit(i, x, G);
            if (u >= wide_items<T>(args) || ld_volatile_shared(wc.abort_flag) != 0) break;
            const PrefillWork w = wide_work<T>(args, u);
            if (w.n_max <= 0) {
                if (T::SPLIT && w.piece >= 0) {
                    // a piece without keys: an empty partial result (merged
                    // as no term) still counts as an arrival
                    const int r = (warp & 3) * 32 + (threadIdx.x & 31);
                    args.part_ml[(size_t)w.piece * 2 * T::BM + r] = -INFINITY;
                    args.part_ml[(size_t)w.piece * 2 * T::BM + T::BM + r] = 0.f;
                    split_arrive<T>(args, w, aux, wc);
                } else {
                    wide_write_empty<T>(args, w);
                }
                continue;
            }
            if (!wide_correction_unit<T>(&tm_o32, args, w, aux, tmem, sQ, wc, J0, kq)) break;
            J0 += w.n_max;
            ++kq;
        }
        // the O stores must have read the staging buffers before exit
        if ((threadIdx.x & 31) == 0) bulk_wait_group_read_0();
        __syncwarp();
    } else {
        setmaxnreg_dec<T::Regs::OTHER>();
        if (warp == T::MMA_WARP)
            wide_mma_role<T>(args, aux, tmem, sQ, sRing, wc, tr);
        else if (warp == T::LOAD_WARP)
            wide_load_role<T>(&tm_q, &tm_k, &tm_v, args, aux, sQ, sRing, wc);
    }

    tc_fence_before();
    __syncthreads();
    if (warp == T::MMA_WARP) {
        tc_fence_after();
        tmem_dealloc(tmem, T::TMEM_COLS);
    }
    // the last piece of a split unit to arrive merges it, on all threads
    if constexpr (SPLIT) {
        if (aux->merge_last != 0 && ld_volatile_shared(wc.abort_flag) == 0)
            merge_unit<T>(args, aux->merge_unit[0], aux->merge_unit[1], aux->merge_unit[2],
                          aux->merge_unit[3], (int)threadIdx.x, T::THREADS);
    }
}

}  // namespace fa
