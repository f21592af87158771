// gdn_tcw.cuh -- the chunk loop with both 64-column halves of d_v = 128 in one
// CTA: one CTA per (sequence, head) instead of two.  Its chunk period is
// longer (≈ 5.3 k cycles against ≈ 4.0 k: the SM carries both halves' register
// work), so it pays where the 64-column loop needs more than one wave of
// CTAs: B8 H16 T4096 d128, 256 CTAs of the 64-column loop against 128 here,
// 0.388 -> 0.290 ms per call.  As a launch of its own (k_gdn_tcw) or in the
// overlapped launch with the chunk prep on the SMs it leaves (k_gdn_tcw_ov).
// Included by gdn_tc.cu inside its namespace (it uses that file's TcParams,
// kC / kNS, the bounded-wait control block and the overlapped launch's prep
// role).  Forward only; dense and packed batches (the overlapped form:
// dense only); d_v a multiple of 128, one CTA per 128-column tile.
//
// The algebra is the chain kernel's ("Gated DeltaNet GPU并行实现", sections
// 3.2-3.3): per chunk, V' = U - W H, O = diag(gamma) Q H + P' V' (P' the
// causal decayed Q K^T over gamma_r), H <- gamma_C H + K^T diag(e) V'.  What
// changes is the split of the work:
//   - warps 0-3 hold d_v columns 0-63 of the fp32 state H = S^T in registers,
//     warps 4-7 columns 64-127 (the same TMEM lanes, the other 64 columns of
//     every accumulator);
//   - the products over d_v are single tcgen05 MMAs with N = 128: [W; Q] H,
//     U = T_u V, K^T V~ and [x; P'] V' (B operands MN-major, two 64-column
//     blocks 8 KB or d_k x 128 B apart);
//   - warp 8 copies (K, W, Q, both V blocks, T_u per stage), warp 9 issues
//     the state's and the output's products, warps 10-11 form the gates and
//     P' (TMEM lanes 64-127), issue the chunk's Gram (thread 320, behind the
//     previous chunk's state and output products in the in-order tensor
//     pipe, as the two issuing warps of the chain kernel order them) and, in
//     chunks whose decay span is too wide for exp(-g_s), scale Q by gamma in
//     place once the Gram has read it.  (One issuing thread for everything
//     put each Gram's issue between H's publication and [W; Q] H: ≈ 5.5 k
//     cycles per chunk.)
// U and dH share 128 TMEM columns: U(j) is read before V'(j) is published,
// dH(j) written after, and U(j + 1) issued only once H(j + 1) is published
// (after dH(j) was read).  The Gram (64), two [W; Q] H / output accumulators
// (2 x 128) and U / dH (128) take 448 of the 512 columns; one P' buffer
// (the next chunk's Gram, which the P' warps wait for, completes after the
// output product that read it).
// A state-only pass (the first pass of a segment scan) needs H alone: Q is
// not copied, and neither the Gram, P' nor the output product is formed, so
// the tensor pipe carries [W; Q] H, U and K^T V~ per chunk.

constexpr int kThreadsW = 384;   // chain warps 0-7, copy warp 8, MMA warp 9, gate / P' warps 10-11

enum {
    W_FULL = 0,                 // + stage: TMA bytes landed (tx + 32 gate lanes)
    W_READY = W_FULL + kNS,     // + stage: the chunk's gates formed
    W_FREE = W_READY + kNS,     // + stage: its MMAs done (commit) and warps 10-11 done with it
    W_PFREE = W_FREE + kNS,     // P' read by the output product (commit)
    W_PREADY,                   // P' written
    W_G,                        // Gram in TMEM (commit)
    W_M34I,                     // the chunk's K^T V~ and output product issued
    W_UW,                       // U in TMEM (commit)
    W_WQ,                       // [W; Q] (or [W; gamma Q]) final in the stage
    W_M2,                       // [W; Q] H done (commit)
    W_VN,                       // V~ and V' (bf16) in shared memory, U read: both halves
    W_M34,                      // dH and the output product done (commit)
    W_HPUB,                     // bf16 H in shared memory, dH read: both halves
    W_DRAIN,                    // MMA issuer drained
    W_DRAIN2,                   // the Gram's issuer drained
    W_COUNT
};

template <int DK>
struct LayW {
    static constexpr int KB = DK / 64;                // 64-column blocks of K / Q / W
    // One input stage (64-row tiles of 128-byte rows, 128-byte swizzled):
    // K blocks, V (two 64-column blocks), per block [W | Q] (a 128-row
    // operand), then T_u (the 8 KB after it are the unread rows of U's
    // 128-row operand).
    static constexpr int OFF_V = KB * 8192;
    static constexpr int OFF_WQ = OFF_V + 16384;
    static constexpr int OFF_TU = OFF_WQ + KB * 16384;
    static constexpr int STAGE = OFF_TU + 8192;
    static constexpr int OFF_H = kNS * STAGE;          // bf16 H: two blocks of DK rows x 128 B
    static constexpr int HBLK = DK * 128;
    static constexpr int OFF_VT = OFF_H + 2 * HBLK;    // V~ (two blocks), then P'
    static constexpr int OFF_P = OFF_VT + 16384;       // [V~ block 1; P'] is the output product's A
    static constexpr int OFF_VN = OFF_P + 8192;        // V' (two blocks)
    static constexpr int GSZ = 5 * 64;                 // g, beta, gamma, exp(-g), beta gamma
    static constexpr int OFF_G = OFF_VN + 16384;       // 2 x GSZ floats
    static constexpr int OFF_GS = OFF_G + 2 * GSZ * 4;  // per stage raw gates: log_alpha, beta
    static constexpr int OFF_BAR = OFF_GS + kNS * 128 * 4;
    static constexpr int OFF_MISC = OFF_BAR + W_COUNT * 8;
    static constexpr int TOTAL = OFF_MISC + 64;
    static constexpr int ALLOC = TOTAL + 1024;
    static_assert(ALLOC <= 227 * 1024, "shared memory budget (wide chunk loop)");
    static_assert(OFF_WQ % 1024 == 0 && OFF_TU % 1024 == 0 && STAGE % 1024 == 0, "align");
    static_assert(OFF_H % 1024 == 0 && OFF_VT % 1024 == 0 && OFF_VN % 1024 == 0, "align");
};

// TMEM columns (512 allocated)
constexpr uint32_t TW_G = 0, TW_M2 = 64, TW_UH = 320;

// SEG: the segment scan's views (k_gdn_tcw); the overlapped launch has none.
template <int DK, bool SEG>
__device__ __forceinline__ void gdn_tcw_body(const CUtensorMap *tm_q, const CUtensorMap *tm_k,
                                             const CUtensorMap *tm_v, const CUtensorMap *tm_t,
                                             const CUtensorMap *tm_w, const TcParams &p,
                                             const int wt, const int h, const int n,
                                             const int nseq) {
    using L = LayW<DK>;
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *sm = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    uint64_t *bar = reinterpret_cast<uint64_t *>(sm + L::OFF_BAR);
    uint32_t *misc = reinterpret_cast<uint32_t *>(sm + L::OFF_MISC);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(misc + 1);
    float *gb = reinterpret_cast<float *>(sm + L::OFF_G);   // [2][GSZ]

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    // this CTA: d_v columns 128 wt .. 128 wt + 127 of (sequence n, head h);
    // tiles wt >= xsplit compute a segment map's linear part instead (v = 0,
    // h0 = identity, the d_k x d_k final state into hT2)
    long long row0 = 0;
    int len = 0, ytok0 = 0, zcoord = 0;
    bool ok_seq = true, head = false;
    int bseq = n;   // the batch row of (n, h) in h0x
    if (p.sm.cu) {
        const int a = __ldg(p.sm.cu + n), b = __ldg(p.sm.cu + n + 1);
        ok_seq = a >= 0 && a <= b && b <= p.sm.T_total;
        if (ok_seq) {
            row0 = (long long)h * p.sm.T_total + a;
            len = b - a;
        }
        ytok0 = a;
        zcoord = h;
    } else if (SEG && p.segs > 0) {
        // segment scan: sequence n = b * segs + segment
        const int b = n / p.segs, sg = n - b * p.segs;
        int t0;
        seg_range(p, sg, t0, len);
        row0 = ((long long)b * p.sm.H + h) * (long long)p.sm.T + t0;
        ytok0 = t0;
        zcoord = b * p.sm.H + h;
        head = p.seg0_full && sg == 0;
        bseq = b;
    } else {
        row0 = ((long long)n * p.sm.H + h) * (long long)p.sm.T;
        len = p.sm.T;
        zcoord = n * p.sm.H + h;
    }
    if (!ok_seq) {
        if (tid == 0) atomicCAS(p.err, 0, kErrBadIndex);
        return;   // before any barrier or TMEM use
    }
    const int nch = (len + kC - 1) / kC;
    const bool lin = wt >= p.xsplit;                              // linear-part CTA
    if (head && lin) return;   // segment 0 from the true h0: no map to form
    // state-only pass (a segment scan's first): no Q, Gram, P' or output product
    const bool so = SEG && p.no_output != 0 && !head;
    const int vx0 = 128 * (lin ? wt - p.xsplit : wt);             // first state column
    const int dvs = lin ? p.dv2 : p.dv;                          // width of this CTA's state
    float *hTp = lin ? p.hT2 : p.hT;
    const long long srow = ((long long)n * p.sm.H + h) * dvs;    // state rows of (n, h)
    // initial state: h0 at (n, h), or for segment 0 run in full h0x at (b, h)
    const float *h0p = head ? p.h0x : p.h0;
    const long long srow0 = head ? ((long long)bseq * p.sm.H + h) * dvs : srow;
    const long long slot0 = p.sm.cu ? (long long)(ytok0 / kC) + n : (long long)n * p.max_chunks;

    if (warp == 9) {
        tmem_alloc(misc, 512);
        tmem_relinquish();
    }
    if (tid == 0) {
        for (int i = 0; i < W_COUNT; ++i) mbar_init(bar + i, 1);
        for (int s = 0; s < kNS; ++s) mbar_init(bar + W_FREE + s, 2);    // MMA commit + warps 10-11
        for (int s = 0; s < kNS; ++s) mbar_init(bar + W_FULL + s, 33);   // TMA tx + 32 gate lanes
        *abort_flag = 0;
        fence_mbar_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = misc[0];
    // T_u and W of the lead chunks come from the launch before this one
    griddep_wait();
    CTA_SPAN(0);
    const Ctl ctl{bar, abort_flag, p.err, p.wait_limit};
    // element counts of the global arrays, for the bounds-check build
    const long long nrows =
        p.sm.cu ? (long long)p.sm.H * p.sm.T_total : (long long)p.sm.N * p.sm.H * p.sm.T;
    const long long nstate = (long long)nseq * p.sm.H * dvs * DK;
    const long long nstate0 = head ? (long long)p.sm.N * p.sm.H * dvs * DK : nstate;
    (void)nrows;
    (void)nstate;
    (void)nstate0;

    if (warp < 8) {
        // ====================================== chain: two halves of d_v
        const int hf = warp >> 2, t = tid & 127;   // TMEM lane = H row (d_k index) / output row - 64
        const int dv0 = vx0 + 64 * hf;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
        float hreg[64];
#pragma unroll
        for (int c = 0; c < 64; ++c)
            hreg[c] = lin ? ((t < DK && dv0 + c == t) ? 1.f : 0.f)
                          : ((t < DK && h0p &&
                              GDN_IDX_OK((srow0 + dv0 + c) * DK + t, 1, nstate0))
                                 ? __ldg(h0p + (srow0 + dv0 + c) * DK + t)
                                 : 0.f);
        uint8_t *Hs = sm + L::OFF_H + hf * L::HBLK;
        uint8_t *VT = sm + L::OFF_VT + hf * 8192, *VN = sm + L::OFF_VN + hf * 8192;
        // Output rows of chunk jj (lanes 64-127 of its accumulator, this
        // half's 64 columns), times osc: gamma_r when the accumulator holds
        // Q H + (P / gamma_r) V' (Q left unscaled), else 1.
        float osc = 1.f;
        auto store_o = [&](int jj) {
            const int r = t - 64;
            const int Lj = min(kC, len - jj * kC);
            uint32_t o0[32], o1[32];
            const uint32_t acc = tmem + lane_base + TW_M2 + (jj & 1) * 128 + 64 * hf;
            tmem_ld32(acc, o0);
            tmem_ld32(acc + 32, o1);
            tmem_wait32(o0);
            tmem_wait32(o1);
            if (r < Lj && GDN_IDX_OK((row0 + (long long)jj * kC + r) * p.dv + dv0, 64,
                                     nrows * p.dv)) {
                uint4 *dst = reinterpret_cast<uint4 *>(p.o + (row0 + (long long)jj * kC + r) *
                                                                 p.dv + dv0);
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[q] = make_uint4(pack_bf16(f32(o0[8 * q]) * osc, f32(o0[8 * q + 1]) * osc),
                                        pack_bf16(f32(o0[8 * q + 2]) * osc, f32(o0[8 * q + 3]) * osc),
                                        pack_bf16(f32(o0[8 * q + 4]) * osc, f32(o0[8 * q + 5]) * osc),
                                        pack_bf16(f32(o0[8 * q + 6]) * osc, f32(o0[8 * q + 7]) * osc));
#pragma unroll
                for (int q = 0; q < 4; ++q)
                    dst[4 + q] =
                        make_uint4(pack_bf16(f32(o1[8 * q]) * osc, f32(o1[8 * q + 1]) * osc),
                                   pack_bf16(f32(o1[8 * q + 2]) * osc, f32(o1[8 * q + 3]) * osc),
                                   pack_bf16(f32(o1[8 * q + 4]) * osc, f32(o1[8 * q + 5]) * osc),
                                   pack_bf16(f32(o1[8 * q + 6]) * osc, f32(o1[8 * q + 7]) * osc));
            }
        };
        bool alive = true;
        for (int j = 0; j < nch; ++j) {
            // (i) publish H as the bf16 B operand of [W; Q] H (dH(j - 1) was
            //     read in the update below: U(j) may now take its columns)
            TRACE(0, j, 0, tid == 0);
            if (t < DK) put_row64(Hs, t, hreg);
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(1, 256);
            if (tid == 0) mbar_arrive(bar + W_HPUB);
            TRACE(0, j, 1, tid == 0);
            // (i') the previous chunk's output rows, off the state's path
            const bool out = !so && !lin;
            if (j > 0 && t >= 64 && out) store_o(j - 1);
            // (ii) V' = U - W H and its decayed copy V~ for the state update
            {
                bool ok = ctl.wait(W_READY + (j % kNS), (j / kNS) & 1);   // this chunk's gates
                ok = ok && ctl.wait(W_UW, j & 1) && ctl.wait(W_M2, j & 1);
                if (!named_bar_and(1, 256, ok)) {
                    alive = false;
                    break;
                }
            }
            TRACE(0, j, 2, tid == 0);
            tc_fence_after();
            const float *gj = gb + (j & 1) * L::GSZ;
            const float gC = gj[63];
            const float decayC = __expf(gC);
            // this chunk's output scale, kept in a register: its gate buffer
            // may be refilled before the rows are stored during chunk j + 1
            const float osc_j = (t >= 64 && gC > -80.f) ? gj[128 + t - 64] : 1.f;
            if (t < 64) {
                const float ev = __expf(gC - gj[t]);
                const uint32_t acc = tmem + lane_base + TW_M2 + (j & 1) * 128 + 64 * hf;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    uint32_t wh[32], u[32];
                    tmem_ld32(acc + 32 * half, wh);
                    tmem_ld32(tmem + lane_base + TW_UH + 64 * hf + 32 * half, u);
                    tmem_wait32(wh);
                    tmem_wait32(u);
                    float vn[32], vt[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        vn[i] = f32(u[i]) - f32(wh[i]);
                        vt[i] = vn[i] * ev;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) {
                        put8(VN, t, 4 * half + q, vn + 8 * q);
                        put8(VT, t, 4 * half + q, vt + 8 * q);
                    }
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(1, 256);
            if (tid == 0) mbar_arrive(bar + W_VN);
            TRACE(0, j, 3, tid == 0);
            // (iii) H <- exp(g_C) H + dH
            if (!named_bar_and(1, 256, ctl.wait(W_M34, j & 1))) {
                alive = false;
                break;
            }
            TRACE(0, j, 4, tid == 0);
            tc_fence_after();
            osc = osc_j;
            if (t < DK) {
                uint32_t d0[32], d1[32];
                tmem_ld32(tmem + lane_base + TW_UH + 64 * hf, d0);
                tmem_ld32(tmem + lane_base + TW_UH + 64 * hf + 32, d1);
                tmem_wait32(d0);
                tmem_wait32(d1);
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    hreg[i] = fmaf(decayC, hreg[i], f32(d0[i]));
                    hreg[32 + i] = fmaf(decayC, hreg[32 + i], f32(d1[i]));
                }
            }
        }
        if (alive && nch > 0 && t >= 64 && !so && !lin) store_o(nch - 1);
        if (alive && hTp && t < DK) {
#pragma unroll
            for (int c = 0; c < 64; ++c)
                if (GDN_IDX_OK((srow + dv0 + c) * DK + t, 1, nstate))
                    hTp[(srow + dv0 + c) * DK + t] = hreg[c];
        }
    } else if (warp == 8) {
        // ================================================= TMA producer
        // lane 0 issues the bulk tensor copies; all lanes stage the chunk's
        // gates (log_alpha, beta; zero past the sequence) next to them
        if (lane == 0) {
            prefetch_tmap(tm_q);
            prefetch_tmap(tm_k);
            prefetch_tmap(tm_v);
            prefetch_tmap(tm_t);
            prefetch_tmap(tm_w);
        }
        int issued = 0;
        float pla0 = 0.f, pla1 = 0.f, pb0 = 0.f, pb1 = 0.f;
        auto load_gates = [&](int jj) {
            const long long r0 = row0 + (long long)jj * kC;
            const int Lj = min(kC, len - jj * kC);
            const bool in0 = lane < Lj && GDN_IDX_OK(r0 + lane, 1, nrows);
            const bool in1 = lane + 32 < Lj && GDN_IDX_OK(r0 + lane + 32, 1, nrows);
            pla0 = in0 ? __ldg(p.log_alpha + r0 + lane) : 0.f;
            pla1 = in1 ? __ldg(p.log_alpha + r0 + lane + 32) : 0.f;
            pb0 = in0 ? __ldg(p.beta + r0 + lane) : 0.f;
            pb1 = in1 ? __ldg(p.beta + r0 + lane + 32) : 0.f;
        };
        if (nch > 0) load_gates(0);
        for (int j = 0; j < nch; ++j) {
            const int s = j % kNS;
            if (p.done && j >= p.prep_c0) {
                // this chunk's T_u and W rows come from the prep CTAs of the
                // same launch: their ready flag
                const bool okp =
                    ctl.gflag(p.done + (long long)h * p.chunk_slots + slot0 + j, 1u);
                if (!__all_sync(0xffffffffu, okp)) break;
                fence_proxy_async_global();
            }
            const bool ok = j < kNS || ctl.wait(W_FREE + s, ((j / kNS) - 1) & 1);
            if (!__all_sync(0xffffffffu, ok)) break;
            uint8_t *stg = sm + s * L::STAGE;
            uint64_t *fb = bar + W_FULL + s;
            const int y = ytok0 + j * kC;
            if (lane == 0) {
                mbar_arrive_expect_tx(fb, (uint32_t)(L::STAGE - (lin ? 16384 : 0) -
                                                     (so ? L::KB * 8192 : 0)));
#pragma unroll
                for (int blk = 0; blk < L::KB; ++blk) {
                    tma_load_3d(stg + blk * 8192, tm_k, fb, blk * 64, y, zcoord);
                    tma_load_3d(stg + L::OFF_WQ + blk * 16384, tm_w, fb, blk * 64, y, zcoord);
                    if (!so)
                        tma_load_3d(stg + L::OFF_WQ + blk * 16384 + 8192, tm_q, fb, blk * 64, y,
                                    zcoord);
                }
                if (!lin) {
                    tma_load_3d(stg + L::OFF_V, tm_v, fb, vx0, y, zcoord);
                    tma_load_3d(stg + L::OFF_V + 8192, tm_v, fb, vx0 + 64, y, zcoord);
                }
                tma_load_3d(stg + L::OFF_TU, tm_t, fb, 0, y, zcoord);
            }
            {
                float *gs = reinterpret_cast<float *>(sm + L::OFF_GS) + s * 128;
                gs[lane] = pla0;
                gs[32 + lane] = pla1;
                gs[64 + lane] = pb0;
                gs[96 + lane] = pb1;
                mbar_arrive(fb);
                if (j + 1 < nch) load_gates(j + 1);
            }
            issued = j + 1;
        }
        // on abort, let copies still in flight land before the CTA exits
        if (lane == 0 && *abort_flag) {
            for (int j = max(0, issued - kNS); j < issued; ++j)
                mbar_wait(bar + W_FULL + j % kNS, (j / kNS) & 1, ctl.limit);
        }
    } else if (warp == 9) {
        // ======================================== MMA issuer (and TMEM owner)
        if (lane == 0 && nch > 0) {
            constexpr uint32_t idN = make_idesc_bf16(128, 128, false, true);    // [W;Q] H, [T_u;x] V, [x;P'] V'
            constexpr uint32_t idKT = make_idesc_bf16(128, 128, true, true);    // K^T V~
            const uint32_t sbase = smem_u32(sm);
            // descriptor bases; an operand at base + off is base_desc + (off >> 4)
            const uint64_t dS = make_sdesc(sbase, 16, 1024, kSwizzle128B);          // K-major, stage
            const uint64_t dKT = make_sdesc(sbase, 8192, 1024, kSwizzle128B);       // K^T, MN-major
            const uint64_t dV = make_sdesc(sbase + L::OFF_V, 8192, 1024, kSwizzle128B);
            const uint64_t dH = make_sdesc(sbase + L::OFF_H, L::HBLK, 1024, kSwizzle128B);
            const uint64_t dVT = make_sdesc(sbase + L::OFF_VT, 8192, 1024, kSwizzle128B);
            const uint64_t dVN = make_sdesc(sbase + L::OFF_VN, 8192, 1024, kSwizzle128B);
            const uint64_t dXP = make_sdesc(sbase + L::OFF_VT + 8192, 16, 1024, kSwizzle128B);
            for (int j = 0; j < nch; ++j) {
                const int s = j % kNS;
                const uint32_t soff = s * L::STAGE;
                const uint32_t acc = tmem + TW_M2 + (j & 1) * 128;
                if (!ctl.wait(W_WQ, j & 1) || !ctl.wait(W_HPUB, j & 1)) break;
                TRACE(2, j, 0, true);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < DK / 16; ++kk) {
                    const uint32_t off = soff + L::OFF_WQ + (kk >> 2) * 16384 + (kk & 3) * 32;
                    mma_bf16(acc, dS + (off >> 4), dH + ((kk * 2048) >> 4), idN, kk > 0);
                }
                mma_commit(bar + W_M2);
                // U = T_u V into the columns dH(j - 1) left (read before H was
                // published); rows 64-127 of the A operand are never read
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk)
                    mma_bf16(tmem + TW_UH, dS + ((soff + L::OFF_TU + kk * 32) >> 4),
                             dV + ((soff + kk * 2048) >> 4), idN, kk > 0);
                mma_commit(bar + W_UW);
                TRACE(2, j, 1, true);
                if (!ctl.wait(W_PREADY, j & 1) || !ctl.wait(W_VN, j & 1)) break;
                TRACE(2, j, 2, true);
                tc_fence_after();
#pragma unroll
                for (int kk = 0; kk < kC / 16; ++kk) {
                    mma_bf16(tmem + TW_UH, dKT + ((soff + kk * 2048) >> 4),
                             dVT + ((kk * 2048) >> 4), idKT, kk > 0);
                    if (!so)
                        mma_bf16(acc, dXP + ((kk * 32) >> 4), dVN + ((kk * 2048) >> 4), idN,
                                 1u);
                }
                mma_commit(bar + W_M34);
                mma_commit(bar + W_PFREE);
                mma_commit(bar + W_FREE + s);
                // the next chunk's Gram (issued by warp 10) goes behind these
                // in the in-order tensor pipe
                mbar_arrive(bar + W_M34I);
                TRACE(2, j, 3, true);
            }
            // every issued MMA has finished before TMEM is released
            mma_commit(bar + W_DRAIN);
            mbar_wait(bar + W_DRAIN, 0, ctl.limit);
        }
    } else {
        // ====================================== gates and P' (warps 10-11)
        const int t = tid - 320, w = warp - 10;
        const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;   // TMEM lanes 64-127
        uint8_t *Pt = sm + L::OFF_P;
        if (lin) {
            // v = 0: the V tiles are never loaded, so clear them once (ordered
            // before the first U product by this chunk's barriers)
            for (int i = t; i < kNS * 1024; i += 64)
                st16(sm + (i >> 10) * L::STAGE + L::OFF_V + (i & 1023) * 16, 0u, 0u, 0u, 0u);
        }
        if (so) {
            // Q is never loaded in a state-only pass: clear its blocks once
            // (ordered before the first [W; Q] H by the W_WQ arrival), so that
            // the product's unread output rows stay finite
            for (int i = t; i < kNS * L::KB * 512; i += 64) {
                const int s = i / (L::KB * 512), r = i - s * (L::KB * 512);
                st16(sm + s * L::STAGE + L::OFF_WQ + (r >> 9) * 16384 + 8192 + (r & 511) * 16,
                     0u, 0u, 0u, 0u);
            }
        }
        if (lin || so) fence_proxy_async_smem();
        for (int j = 0; j < nch; ++j) {
            const int s = j % kNS;
            uint8_t *stg = sm + s * L::STAGE;
            float *gj = gb + (j & 1) * L::GSZ;
            if (!named_bar_and(4, 64, ctl.wait(W_FULL + s, (j / kNS) & 1))) break;
            TRACE(1, j, 0, t == 0);
            if (w == 0) {
                const float *gs = reinterpret_cast<const float *>(sm + L::OFF_GS) + s * 128;
                float la0 = gs[lane], la1 = gs[32 + lane];
                const float b0 = gs[64 + lane], b1 = gs[96 + lane];
#pragma unroll
                for (int off = 1; off < 32; off <<= 1) {
                    const float y0 = __shfl_up_sync(0xffffffffu, la0, off);
                    const float y1 = __shfl_up_sync(0xffffffffu, la1, off);
                    if (lane >= off) {
                        la0 += y0;
                        la1 += y1;
                    }
                }
                la1 += __shfl_sync(0xffffffffu, la0, 31);
                const float e0 = __expf(la0), e1 = __expf(la1);
                gj[lane] = la0;
                gj[lane + 32] = la1;
                gj[64 + lane] = b0;
                gj[64 + lane + 32] = b1;
                gj[128 + lane] = e0;
                gj[128 + lane + 32] = e1;
                gj[192 + lane] = __expf(-la0);   // used only when the span is < 80
                gj[192 + lane + 32] = __expf(-la1);
                gj[256 + lane] = b0 * e0;
                gj[256 + lane + 32] = b1 * e1;
            }
            const int L_ = min(kC, len - j * kC);
            if (p.sm.cu && L_ < kC) {
                // rows past this sequence belong to the next one: clear them in
                // every tile of the stage (K, W, Q, both V blocks, T_u)
                constexpr int per_row = 3 * DK / 8 + 24;   // 16-byte pieces per row
                for (int i = t; i < (kC - L_) * per_row; i += 64) {
                    const int r = L_ + i / per_row, q = i % per_row;
                    uint8_t *base;
                    if (q < DK / 8)   // K
                        base = stg + (q >> 3) * 8192;
                    else if (q < 3 * DK / 8)   // W, Q blocks
                        base = stg + L::OFF_WQ + ((q - DK / 8) >> 3) * 8192;
                    else if (q < 3 * DK / 8 + 16)   // V blocks
                        base = stg + L::OFF_V + ((q - 3 * DK / 8) >> 3) * 8192;
                    else   // T_u
                        base = stg + L::OFF_TU;
                    st16(base + sw128_offset(r, q & 7), 0u, 0u, 0u, 0u);
                }
                fence_proxy_async_smem();
            }
            named_bar(4, 64);
            if (t == 0) mbar_arrive(bar + W_READY + s);
            const bool span_ok = gj[63] > -80.f;
            // [W; Q] for the chain MMA: now when Q stays unscaled (the output
            // rows take gamma_r at the end, P' is formed divided by gamma_r),
            // once the previous chunk's chain MMA has read its own copy (the
            // mbarrier then never runs two phases ahead of its waiter)
            if (span_ok || so) {
                if (!named_bar_and(4, 64, j == 0 || ctl.wait(W_M2, (j - 1) & 1))) break;
                if (t == 0) mbar_arrive(bar + W_WQ);
            }
            // this chunk's Gram [W; Q] K^T (its Q rows give P'), behind the
            // previous chunk's state and output products (the G(j - 1) rows
            // were read above, before the last barrier)
            if (t == 0 && !so) {
                if (j == 0 || ctl.wait(W_M34I, (j - 1) & 1)) {
                    tc_fence_after();
                    const uint32_t sbase = smem_u32(sm), soff = s * L::STAGE;
                    const uint64_t dS = make_sdesc(sbase, 16, 1024, kSwizzle128B);
                    constexpr uint32_t idG = make_idesc_bf16(128, 64, false, false);
#pragma unroll
                    for (int kk = 0; kk < DK / 16; ++kk) {
                        const uint32_t kof = soff + (kk >> 2) * 8192 + (kk & 3) * 32;
                        const uint32_t aof = soff + L::OFF_WQ + (kk >> 2) * 16384 + (kk & 3) * 32;
                        mma_bf16(tmem + TW_G, dS + (aof >> 4), dS + (kof >> 4), idG, kk > 0);
                    }
                    mma_commit(bar + W_G);
                }
            }
            // P' from the Gram's Q rows, once the previous P' was read
            // (a state-only pass forms neither: the P' barriers still pace
            // these warps one chunk ahead of the issuer at most)
            bool okg = so || ctl.wait(W_G, j & 1);
            if (j > 0) okg = okg && ctl.wait(W_PFREE, (j - 1) & 1);
            if (!named_bar_and(4, 64, okg)) break;
            TRACE(1, j, 2, t == 0);
            tc_fence_after();
            if (!so) {
                const int r = t;
                uint32_t g0[32], g1[32];
                tmem_ld32(tmem + lane_base + TW_G, g0);
                tmem_ld32(tmem + lane_base + TW_G + 32, g1);
                const float gr = gj[r];
                tmem_wait32(g0);
                tmem_wait32(g1);
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    float x[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        const int sidx = 32 * half + i;
                        const float gv = f32(half == 0 ? g0[i] : g1[i]);
                        const bool keep = sidx <= r;
                        const float f = span_ok ? gj[192 + sidx]
                                                : __expf(keep ? gr - gj[sidx] : 0.f);
                        x[i] = keep ? f * gv : 0.f;
                    }
#pragma unroll
                    for (int q = 0; q < 4; ++q) put8(Pt, r, 4 * half + q, x + 8 * q);
                }
            }
            fence_proxy_async_smem();
            tc_fence_before();
            named_bar(4, 64);
            if (t == 0) mbar_arrive(bar + W_PREADY);
            TRACE(1, j, 3, t == 0);
            if (!span_ok && !so) {
                // the Gram has read Q: gamma Q in place (row t of every Q
                // block: loads first, then stores), then [W; gamma Q]
                const float gam = gj[128 + t];
#pragma unroll
                for (int blk = 0; blk < L::KB; ++blk) {
                    uint8_t *qs = stg + L::OFF_WQ + blk * 16384 + 8192;
                    uint4 v[8];
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        v[ch] = *reinterpret_cast<const uint4 *>(qs + sw128_offset(t, ch));
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch) {
                        uint32_t wv[4] = {v[ch].x, v[ch].y, v[ch].z, v[ch].w};
#pragma unroll
                        for (int e = 0; e < 4; ++e) {
                            __nv_bfloat162 b2 = *reinterpret_cast<__nv_bfloat162 *>(&wv[e]);
                            float2 f2 = __bfloat1622float2(b2);
                            wv[e] = pack_bf16(f2.x * gam, f2.y * gam);
                        }
                        v[ch] = make_uint4(wv[0], wv[1], wv[2], wv[3]);
                    }
#pragma unroll
                    for (int ch = 0; ch < 8; ++ch)
                        if (GDN_SMEM_OK(smem_u32(qs + sw128_offset(t, ch)), 16))
                            *reinterpret_cast<uint4 *>(qs + sw128_offset(t, ch)) = v[ch];
                }
                fence_proxy_async_smem();
                if (!named_bar_and(4, 64, j == 0 || ctl.wait(W_M2, (j - 1) & 1))) break;
                if (t == 0) mbar_arrive(bar + W_WQ);
            }
            if (t == 0) mbar_arrive(bar + W_FREE + s);
        }
        // every Gram issued here has finished before TMEM is released
        if (t == 0 && nch > 0 && !so) {
            mma_commit(bar + W_DRAIN2);
            mbar_wait(bar + W_DRAIN2, 0, ctl.limit);
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    CTA_SPAN(1);
    if (warp == 9) tmem_dealloc(tmem, 512);
}

// The wide chunk loop alone, one CTA per (sequence, head, 128-column d_v
// tile) (the chunk prep ran before it, as one launch); dense or packed.
template <int DK>
__global__ void __launch_bounds__(kThreadsW, 1)
k_gdn_tcw(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_t,
          const __grid_constant__ CUtensorMap tm_w, TcParams p) {
    // block b: tile b % tiles of head (b / tiles) % H of sequence b / (tiles H);
    // in a segment scan the sequences run segment-major (segment seg_lo of
    // every batch row first), so the longest CTAs start in the first wave
    const int tiles = p.xsplit + p.lin_tiles, b = (int)blockIdx.x, hn = b / tiles;
    const int h = hn % p.sm.H, q = hn / p.sm.H;
    if (p.segs > 0) {
        const int sg = p.seg_lo + q / p.sm.N, bb = q - (q / p.sm.N) * p.sm.N;
        gdn_tcw_body<DK, true>(&tm_q, &tm_k, &tm_v, &tm_t, &tm_w, p, b - hn * tiles, h,
                               bb * p.segs + sg, p.sm.N * p.segs);
    } else {
        // a packed batch may run its sequences in a given order (longest first)
        const int n = p.seq_order ? __ldg(p.seq_order + q) : q;
        gdn_tcw_body<DK, true>(&tm_q, &tm_k, &tm_v, &tm_t, &tm_w, p, b - hn * tiles, h, n,
                               gridDim.x / (tiles * p.sm.H));
    }
}

// The overlapped launch with the wide chunk loop: roles below nchain (one per
// (sequence, head)) run gdn_tcw_body, the others the chunk prep.
template <int DK>
__global__ void __launch_bounds__(kThreadsW, 1)
k_gdn_tcw_ov(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
             const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_t,
             const __grid_constant__ CUtensorMap tm_w, TcParams p, UtParams up, int nchain,
             int by_sm) {
    const int role = ov_role(by_sm);
    if (role < nchain) {
        const int tiles = p.xsplit, hn = role / tiles;
        gdn_tcw_body<DK, false>(&tm_q, &tm_k, &tm_v, &tm_t, &tm_w, p, role - hn * tiles,
                                hn % p.sm.H, hn / p.sm.H, p.sm.N);
        return;
    }
    ov_prep_role<DK>(&tm_k, up, role, nchain);
}
