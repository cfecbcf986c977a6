// Short-row pipelined kernel: forward and verify-ring passes over rows of a
// few tokens -- speculative-decoding verify windows
// ("gated_delta_recurrence_verify_ring_gpu").  (Snapshot passes run on the
// general kernel, which stores snapshots straight from registers.)
//
// Persistent CTAs walk (row, value head, CW-column tile) units like the
// pipelined decode kernel.  A unit's stage holds the bf16/f32 state tile and
// the operands of its first TCH tokens, all copied with cp.async while the
// previous unit computes.  The tile is widened into float32 registers once
// and stays there for the whole row: lane kl = lane % LK holds RG (even)
// consecutive 8-row groups in the row-pair form of gdr_state.cuh, lane
// vl = lane / LK holds 2 columns.  With bf16 pools LK = 4 (32 rows per lane),
// with float32 pools RG = 2; the in-thread tree levels are adds and the rest a
// butterfly over the LK lanes.  For each staged chunk the CTA's warps first
// normalise the tokens (q~, k^ pair-interleaved, alpha and k^.q~ written back
// into the stage; ring records get k^ and alpha here), then every warp runs
// the chunk's tokens on its columns with warp shuffles only.  The final commit
// goes back through the stage and leaves the SM as coalesced rows.  Rows longer than
// TCH load further chunks in place.  The arithmetic is the fixed sequence of
// gdr_device.cuh, so results equal the other kernels' bit for bit.
#include "gdr_pipe.cuh"
#include "gdr_state.cuh"

namespace gdr {

// Tile width of the short-row kernel (kShortTileWarps x 16 columns), lanes
// along K for bf16 pools (the warps per CTA follow: tile width / (32 / LK x 2
// columns)), and CTAs per SM it is compiled for.
constexpr int kShortTileWarps = 4;
constexpr int kShortLKbf16 = 4;
constexpr int kShortMinBlocksBf16 = 4;
constexpr int kShortMinBlocksF32 = 4;

// Tile swizzle shift: a lane owns 16 (f32) or 32 (bf16) consecutive rows, so
// the row's 16-row block picks the chunk permutation (conflict-free reads).
constexpr int kShortSwizzle = 4;

template <typename ST, int K> using ShortTile = PipeShape<ST, K, kShortTileWarps>;

template <typename ST, int K> struct WinShape {
    using P = ShortTile<ST, K>;                          // tile geometry (CW, CPR, S_STATE, USL)
    static constexpr bool BF = sizeof(ST) == 2;
    static constexpr int NG = K / 8;
    static constexpr int LK = BF ? cmin(kShortLKbf16, K / 16) : K / 16;  // lanes along K
    static constexpr int RG = NG / LK;                   // 8-row groups per lane (even)
    static constexpr int ROWS = 8 * RG;
    static constexpr int LV = 32 / LK;
    static constexpr int C = 2;                          // columns per lane
    static constexpr int WC = LV * C;
    static constexpr int NW = P::CW / WC;                // warps per CTA
    static constexpr int NT = 32 * NW;
    static constexpr int KP = K + LK * 4;                // floats per staged q / k vector (padded)
    static constexpr int TQ = KP / 4, TV = P::CW / 4;    // 16-byte chunks
    static constexpr int TOKV = 2 * TQ + TV;
    static constexpr int TOK = TOKV + 1;                 // + {decay -> alpha, beta, k^.q~, -}
    static constexpr int TCH = 8;                        // tokens per staged chunk
    static constexpr int SC = P::S_STATE + TCH * TOK;    // chunks per stage
    static constexpr int SMEM1 = SC * 16;
    static constexpr int NL = NG / 2;                    // lanes per token when normalising
    static constexpr int TPW = 32 / NL;                  // tokens per warp when normalising
    static constexpr int MINB = BF ? kShortMinBlocksBf16 : kShortMinBlocksF32;  // CTAs per SM
    using State = LaneState<RG, C>;
    static_assert(RG % 2 == 0, "row-pair form");
};

// Float offset of raw row i inside a staged q / k vector.
template <typename ST, int K> __device__ __forceinline__ int tpos(int i) {
    return vpos<false, WinShape<ST, K>::ROWS>(i);
}

// A unit of the short kernel: row b, value head h (key head hk, index jr
// inside its GQA group), tile us.  Past the end of the batch: an empty row.
struct ShortMeta {
    int b, h, hk, jr, us, t0, t1, slot;
};

// Unit index u -> (b, h, us), us fastest; hd divides by nv * USL, rd by r.
template <int USL>
__device__ __forceinline__ ShortMeta short_meta(const StepParams &p, long long u, int nunits, FastDiv hd,
                                                FastDiv rd) {
    ShortMeta m{};
    if (u >= nunits) return m;
    const unsigned ui = (unsigned)u;
    m.b = (int)hd.div(ui);
    const int hu = (int)(ui - (unsigned)m.b * hd.d);
    m.h = hu / USL;
    m.us = hu % USL;
    m.hk = (int)rd.div((unsigned)m.h);
    m.jr = m.h - m.hk * p.r;
    m.t0 = p.offsets[m.b];
    m.t1 = p.offsets[m.b + 1];
    m.slot = p.slot_idx[m.b];
    return m;
}

__device__ __forceinline__ bool short_unit_valid(const StepParams &p, const ShortMeta &m, long long max_len) {
    const int L = m.t1 - m.t0;
    return m.t0 >= 0 && L >= 1 && m.t1 <= p.T && (max_len <= 0 || L <= max_len) && m.slot >= 0 &&
           m.slot < p.max_slots;
}

// Queue the operands of tokens [cb, cb + tc) of the unit's row.  Thread
// r < RV copies 16-byte chunk r of every token (raw q, raw k, then the tile's
// v columns); threads RV .. RV + tc - 1 copy one token's decay and beta.
template <typename ST, int K>
__device__ __forceinline__ void short_issue_tokens(const StepParams &p, const ShortMeta &m, int cb, int tc,
                                                   uint4 *stage) {
    using W = WinShape<ST, K>;
    using P = ShortTile<ST, K>;
    constexpr int RQ = K / 4;  // raw chunks per q / k vector
    constexpr int RV = 2 * RQ + W::TV;
    static_assert(RV + W::TCH <= W::NT, "one chunk role per thread");
    const int r = threadIdx.x;
    uint4 *tok = stage + P::S_STATE;
    if (r < RV) {
        int src, dst;
        if (r < RQ) {
            src = m.hk * K + 4 * r;
            dst = tpos<ST, K>(4 * r) / 4;
        } else if (r < 2 * RQ) {
            src = (p.nk + m.hk) * K + 4 * (r - RQ);
            dst = W::TQ + tpos<ST, K>(4 * (r - RQ)) / 4;
        } else {
            src = 2 * p.nk * K + m.h * K + m.us * P::CW + 4 * (r - 2 * RQ);
            dst = 2 * W::TQ + (r - 2 * RQ);
        }
        const float *g = p.qkv + (long long)(m.t0 + cb) * p.qkv_ss + src;
        uint4 *d = tok + dst;
        for (int tt = 0; tt < tc; ++tt, g += p.qkv_ss, d += W::TOK) cp_async16(d, g);
    } else if (r < RV + tc) {
        const int tt = r - RV;
        float *ab = reinterpret_cast<float *>(tok + tt * W::TOK + W::TOKV);
        const long long o = (long long)(m.t0 + cb + tt) * p.tok_ss + (long long)m.h * p.tok_hs;
        cp_async4(ab, p.decay + o);
        cp_async4(ab + 1, p.beta + o);
    }
}

template <typename ST, int K>
__device__ __forceinline__ void short_issue(const StepParams &p, const ShortMeta &m, long long max_len,
                                            uint4 *stage) {
    using P = ShortTile<ST, K>;
    using W = WinShape<ST, K>;
    if (short_unit_valid(p, m, max_len)) {
        tile_issue<ST, K, W::NT, kShortTileWarps, kShortSwizzle>(reinterpret_cast<const ST *>(p.state) + (long long)m.slot * p.st_slot +
                                     (long long)m.h * p.st_head + m.us * P::CW,
                                 p.st_k, stage);
        const int L = m.t1 - m.t0;
        short_issue_tokens<ST, K>(p, m, 0, L < W::TCH ? L : W::TCH, stage);
    }
    cp_async_commit();
}

// This lane's C columns of tile row r (rows keep the 16-byte chunk swizzle).
template <typename ST, int K>
__device__ __forceinline__ ST *tile_cols(uint4 *tile, int r, int col) {
    using P = ShortTile<ST, K>;
    constexpr int EPC = 16 / (int)sizeof(ST);
    return reinterpret_cast<ST *>(tile + r * P::CPR + ((col / EPC) ^ ((r >> kShortSwizzle) & (P::CPR - 1)))) +
           (col % EPC);
}

// The lane's rows in the tile: the 8 rows of a group share the swizzle, so
// each group is one base pointer plus i * CW elements.
template <typename ST, int K>
__device__ __forceinline__ void short_get_tile(uint4 *tile, int r0, int col, typename WinShape<ST, K>::State &s) {
    using W = WinShape<ST, K>;
    constexpr int C = W::C, CW = ShortTile<ST, K>::CW;
#pragma unroll
    for (int g = 0; g < W::RG; ++g) {
        const ST *gb = tile_cols<ST, K>(tile, r0 + 8 * g, col);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            Pack<ST, C> x;
            x.load(gb + i * CW);
#pragma unroll
            for (int c = 0; c < C; ++c) s.set(8 * g + i, c, x.get(c));
        }
    }
}

// Writes the float32 state s (this lane's ROWS rows x C columns) into the tile.
template <typename ST, int K>
__device__ __forceinline__ void short_put_tile(uint4 *tile, int r0, int col, const typename WinShape<ST, K>::State &s) {
    using W = WinShape<ST, K>;
    constexpr int C = W::C, CW = ShortTile<ST, K>::CW;
#pragma unroll
    for (int g = 0; g < W::RG; ++g) {
        ST *gb = tile_cols<ST, K>(tile, r0 + 8 * g, col);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            Pack<ST, C> x;
#pragma unroll
            for (int c = 0; c < C; ++c) x.set(c, s.get(8 * g + i, c));
            x.store(gb + i * CW);
        }
    }
}

// Computes one unit; returns true when the state must be committed (the new
// tile is then in the stage, to be stored by the caller after a barrier).
// Every branch that decides between barriers is uniform over the CTA.
template <typename ST, int K, Mode MODE>
__device__ __forceinline__ bool short_compute(const StepParams &p, const RingParams &rp, const SnapParams &sp,
                                              long long max_len, const ShortMeta &m, uint4 *stage) {
    using P = ShortTile<ST, K>;
    using W = WinShape<ST, K>;
    constexpr int V = K, LK = W::LK, ROWS = W::ROWS, C = W::C, NW = W::NW;
    constexpr int TCH = W::TCH, NL = W::NL, TPW = W::TPW;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kl = lane % LK, vl = lane / LK;
    const int h = m.h, us = m.us, jr = m.jr;
    const bool leader = tid == 0 && h == 0 && us == 0;
    if (m.t0 < 0 || m.t1 < m.t0 || m.t1 > p.T) {
        if (leader) flag(p.status, GDR_STATUS_BAD_OFFSETS);
        return false;
    }
    const int L = m.t1 - m.t0;
    if (L == 0) return false;
    const int col = warp * W::WC + vl * C;  // inside the unit's tile
    float *optr = p.out + (long long)m.t0 * p.out_ss + (long long)(h * V + us * P::CW + col) * p.out_vs;
    if (max_len > 0 && L > max_len) {  // longer than the caller's bound: zero output, nothing else
        if (leader) flag(p.status, GDR_STATUS_ROW_TOO_LONG);
        if (kl == 0) zero_rows<C>(optr, L, p);
        return false;
    }
    if (m.slot < 0 || m.slot >= p.max_slots) {
        if (m.slot != -1 && leader) flag(p.status, GDR_STATUS_BAD_SLOT);
        if (kl == 0) zero_rows<C>(optr, L, p);
        return false;
    }
    // Verify: rows of at most ring_len tokens record and leave the pool alone.
    bool records = false, commit = true;
    long long ring_row = 0;  // element index of this (ring row, key head)'s first record
    if constexpr (MODE == Mode::Verify) {
        if (L <= rp.len) {
            commit = false;
            const int rs = rp.ring_slot[m.b];
            if (rs < 0 || rs >= rp.rows) {
                if (leader) flag(p.status, GDR_STATUS_BAD_RING_SLOT);
            } else {
                records = true;
                ring_row = ((long long)rs * p.nk + m.hk) * rp.len * rp.stride;
            }
        }
    }

    const int r0 = kl * ROWS;  // this lane's first tile row
    typename W::State s;
    short_get_tile<ST, K>(stage, r0, col, s);
    float *tokf = reinterpret_cast<float *>(stage + P::S_STATE);
    // lanes kl == 0 write the output (and u records) of their C columns
    const bool w_out = kl == 0;
    long long uidx = ring_row + rp.u_off + jr * V + us * P::CW + col;  // this lane's u record
    const bool rec_alpha = records && us == 0;
    const bool rec_k = rec_alpha && jr == 0;

    for (int cb = 0; cb < L; cb += TCH) {
        const int tc = min(TCH, L - cb);
        if (cb > 0) {  // a longer row: bring in its next chunk of operands
            __syncthreads();
            short_issue_tokens<ST, K>(p, m, cb, tc, stage);
            cp_async_commit();
            cp_async_wait<0>();
            __syncthreads();
        }
        // normalise: NL lanes per token, TPW tokens per warp, packed into the
        // low warps (a warp with no token skips the pass)
        for (int tb = 0; tb < tc; tb += NW * TPW) {
            if (tb + TPW * warp >= tc) continue;  // uniform over the warp
            const int tt = tb + TPW * warp + lane / NL;
            const bool act = tt < tc;
            float *tq = tokf + (act ? tt : 0) * W::TOK * 4;
            const long long rec = ring_row + (long long)(cb + (act ? tt : 0)) * rp.stride;
            float *ab = tq + W::TOKV * 4;
            norm_token<K, true, ROWS>(tq, tq + W::KP, ab + 2, lane % NL, act, p, rec_k ? rp.ring : nullptr, rp.bf16,
                                      rec);
            if (act && lane % NL == 0) {
                const float alpha = gdr_alpha(ab[0], p.decay_is_log);
                ab[0] = alpha;
                if (rec_alpha) ring_put1(rp.ring, rp.bf16, rec + rp.alpha_off + jr, alpha);
            }
        }
        __syncthreads();

        const float *tq = tokf;  // operands of token cb + tt, advanced per token
        const int base = tpos<ST, K>(r0);  // this lane's run of rows in the staged vectors
        for (int tt = 0; tt < tc; ++tt, tq += W::TOK * 4) {
            const float *tk = tq + W::KP;
            const float *ab = tq + W::TOKV * 4;
            const float alpha = ab[0], beta = ab[1], kq = ab[2];
            float a[C], bq[C];
            s.partials(tk + base, tq + base, a, bq);
            // S <- alpha S now, independent of the reductions' tree; a verify
            // row that does not commit never reads the state after its last token
            const bool adv = commit || cb + tt + 1 < L;
            if (adv) s.scale(alpha);
            const float *tv = tq + 2 * W::KP;
            float u[C], o[C];
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const float A = tree_lanes<LK>(a[c]);
                const float B = tree_lanes<LK>(bq[c]);
                u[c] = gdr_u(beta, alpha, A, tv[col + c]);
                o[c] = gdr_o(alpha, B, kq, u[c]);
            }
            if (w_out) {
                store_f32<C>(optr, p.out_vs, p.out_vec, o);
                if (records) {
                    static_assert(C == 2, "u records are written as pairs");
                    ring_put2(rp.ring, rp.bf16, uidx, u[0], u[1]);
                }
            }
            optr += p.out_ss;
            uidx += rp.stride;
            // S <- k^ u^T + S
            if (adv) s.add_outer(tk + base, u);
        }
    }
    if (commit) short_put_tile<ST, K>(stage, r0, col, s);
    return commit;
}

template <typename ST, int K, Mode MODE>
__global__ void __launch_bounds__(WinShape<ST, K>::NT, WinShape<ST, K>::MINB)
    k_short(const StepParams p, const RingParams rp, const SnapParams sp, const long long max_len,
            const int nunits, const FastDiv hd, const FastDiv rd) {
    using P = ShortTile<ST, K>;
    using W = WinShape<ST, K>;
    extern __shared__ uint4 smem_short[];
    uint4 *stage0 = smem_short, *stage1 = smem_short + W::SC;
    // descriptors of units i, i+1, i+2 (slot i % 3 holds unit i), computed by
    // thread 0 two units ahead and published by the barrier that follows
    __shared__ ShortMeta meta_s[3];
    const long long G = gridDim.x;
    if (threadIdx.x == 0) {
        meta_s[0] = short_meta<P::USL>(p, blockIdx.x, nunits, hd, rd);
        meta_s[1] = short_meta<P::USL>(p, (long long)blockIdx.x + G, nunits, hd, rd);
    }
    __syncthreads();
    short_issue<ST, K>(p, meta_s[0], max_len, stage0);
    int sel = 0, mi = 0;
    for (long long u = blockIdx.x; u < nunits; u += G) {
        uint4 *s_cur = sel ? stage1 : stage0;
        uint4 *s_nxt = sel ? stage0 : stage1;
        const int m1 = mi == 2 ? 0 : mi + 1, m2 = m1 == 2 ? 0 : m1 + 1;
        short_issue<ST, K>(p, meta_s[m1], max_len, s_nxt);
        if (threadIdx.x == 0) meta_s[m2] = short_meta<P::USL>(p, u + 2 * G, nunits, hd, rd);
        cp_async_wait<1>();
        __syncthreads();
        const bool commit = short_compute<ST, K, MODE>(p, rp, sp, max_len, meta_s[mi], s_cur);
        __syncthreads();
        if (commit) {  // uniform over the CTA
            const ShortMeta &cur = meta_s[mi];
            tile_store<ST, K, W::NT, kShortTileWarps, kShortSwizzle>(reinterpret_cast<ST *>(p.state) + (long long)cur.slot * p.st_slot +
                                         (long long)cur.h * p.st_head + cur.us * P::CW,
                                     p.st_k, s_cur);
            __syncthreads();  // the stage is refilled next iteration
        }
        sel ^= 1;
        mi = m1;
    }
    cp_async_wait<0>();
}

template <typename ST, int K, Mode MODE>
static cudaError_t launch_short_m(const StepParams &p, const RingParams &rp, const SnapParams &sp,
                                  long long max_len, cudaStream_t st) {
    using P = ShortTile<ST, K>;
    using W = WinShape<ST, K>;
    constexpr int SMEM = 2 * W::SMEM1;
    static LaunchCache cache;
    LaunchInfo li;
    cudaError_t e = launch_info(cache, &li, [](LaunchInfo &x) {
        cudaError_t r = cudaFuncSetAttribute(k_short<ST, K, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (r != cudaSuccess) return r;
        return cudaOccupancyMaxActiveBlocksPerMultiprocessor(&x.occ, k_short<ST, K, MODE>, W::NT, SMEM);
    });
    if (e != cudaSuccess) return e;
    const long long nunits = (long long)p.batch * p.nv * P::USL;
    long long grid = (long long)li.sms * li.occ;
    if (grid > nunits) grid = nunits;
    if (grid > 0)
        k_short<ST, K, MODE><<<(unsigned)grid, W::NT, SMEM, st>>>(p, rp, sp, max_len, (int)nunits,
                                                                  FastDiv((unsigned)(p.nv * P::USL)),
                                                                  FastDiv((unsigned)p.r));
    return cudaGetLastError();
}

template <typename ST, int K> struct ShortOK {
    static constexpr bool value = ShortTile<ST, K>::OK && WinShape<ST, K>::NT % ShortTile<ST, K>::CPR == 0 &&
                                  ShortTile<ST, K>::S_STATE % WinShape<ST, K>::NT == 0 &&
                                  WinShape<ST, K>::NW >= 1;
};

template <typename ST, int K>
static cudaError_t launch_short_t(const StepParams &p, Mode mode, const RingParams &rp, const SnapParams &sp,
                                  long long max_len, cudaStream_t st, bool *used) {
    *used = false;
    if constexpr (ShortOK<ST, K>::value) {
        if (!p.qkv_vec || (long long)p.batch * p.nv * ShortTile<ST, K>::USL >= (1ll << 31)) return cudaSuccess;
        *used = true;
        switch (mode) {
            case Mode::Fwd: return launch_short_m<ST, K, Mode::Fwd>(p, rp, sp, max_len, st);
            case Mode::Verify: return launch_short_m<ST, K, Mode::Verify>(p, rp, sp, max_len, st);
            case Mode::Snap: *used = false; return cudaSuccess;  // the general kernel takes snapshots
        }
    }
    return cudaSuccess;
}

cudaError_t launch_short(const StepParams &p, int K, bool bf16, Mode mode, const RingParams &rp,
                         const SnapParams &sp, long long max_row_len, cudaStream_t s, bool *used) {
#define GDR_CASE(KK)                                                                            \
    case KK:                                                                                    \
        return bf16 ? launch_short_t<uint16_t, KK>(p, mode, rp, sp, max_row_len, s, used)      \
                    : launch_short_t<float, KK>(p, mode, rp, sp, max_row_len, s, used);
    switch (K) {
        GDR_CASE(16)
        GDR_CASE(32)
        GDR_CASE(64)
        GDR_CASE(128)
    }
#undef GDR_CASE
    *used = false;
    return cudaSuccess;
}

}  // namespace gdr
