// Short-row pipelined kernel: forward, verify-ring and snapshot passes over
// rows of a few tokens -- speculative-decoding verify windows
// ("gated_delta_recurrence_verify_ring_gpu") and Gated Delta Product draft
// sequences ("core.ssm.ops.gdp.fused_recurrent", intermediate_states).
//
// Persistent CTAs walk (row, value head, CW-column tile) units like the
// pipelined decode kernel.  A unit's stage holds the bf16/f32 state tile and
// the operands of its first TCH tokens, all copied with cp.async while the
// previous unit computes.  The tile is widened into float32 registers once
// and stays there for the whole row: lane kl = lane % LK holds RG consecutive
// 8-row groups, lane vl = lane / LK holds C columns.  With bf16 pools LK = 4
// (32 rows x 2 columns per lane), so two of a token's tree levels are
// in-thread adds and the rest is a 4-lane reduce-scatter.  For each staged
// chunk the CTA's warps first normalise one token each (q~, k^, alpha and
// k^.q~ written back into the stage), then every warp runs the chunk's tokens
// on its columns with warp shuffles only.  Snapshots and the final commit go
// back through the stage and leave the SM as coalesced rows.  Rows longer than
// TCH load further chunks in place.  The arithmetic is the fixed sequence of
// gdr_device.cuh, so results equal the other kernels' bit for bit.
#include "gdr_pipe.cuh"

namespace gdr {

// Warps per CTA budget of the short-row kernel (tile width = warps x 16 columns)
// and CTAs per SM it is compiled for.
constexpr int kShortWarps = 4;
constexpr int kShortMinBlocks = 4;

template <typename ST, int K> using ShortTile = PipeShape<ST, K, kShortWarps>;

template <typename ST, int K> struct WinShape {
    using P = ShortTile<ST, K>;                          // tile geometry (CW, CPR, S_STATE, USL)
    static constexpr bool BF = sizeof(ST) == 2;
    static constexpr int LK = BF ? cmin(4, K / 8) : P::LK;  // lanes along K
    static constexpr int RG = K / 8 / LK;                // 8-row groups per lane
    static constexpr int ROWS = 8 * RG;
    static constexpr int LV = 32 / LK;
    static constexpr int C = BF ? 2 : P::C;              // columns per lane
    static constexpr int WC = LV * C;
    static constexpr int NW = P::CW / WC;                // warps per CTA
    static constexpr int NT = 32 * NW;
    static constexpr bool PAD = LK <= 4;                 // pad staged vectors per lane run
    static constexpr int KP = PAD ? K + LK * 4 : K;      // floats per staged q / k vector
    static constexpr int TQ = KP / 4, TV = P::CW / 4;    // 16-byte chunks
    static constexpr int TOKV = 2 * TQ + TV;
    static constexpr int TOK = TOKV + 1;                 // + {decay -> alpha, beta, k^.q~, -}
    static constexpr int TCH = 8;                        // tokens per staged chunk
    static constexpr int SC = P::S_STATE + TCH * TOK;    // chunks per stage
    static constexpr int SMEM1 = SC * 16;
};

// Float offset of row i inside a staged q / k vector (4 spare floats after each
// lane's run of rows keep the LK distinct 16-byte reads in different banks).
template <typename ST, int K> __device__ __forceinline__ int tpos(int i) {
    using W = WinShape<ST, K>;
    if constexpr (W::PAD) return i + (i / W::ROWS) * 4;
    return i;
}

// A unit of the short kernel: hu = h * USL + us; b = row.  Past the end of
// the batch: an empty row.
struct ShortMeta {
    int hu, b, t0, t1, slot;
};

template <int USL>
__device__ __forceinline__ ShortMeta short_meta(const StepParams &p, long long u, int nunits) {
    ShortMeta m{};
    if (u >= nunits) return m;
    const int ui = (int)u;
    const int bh = ui / USL;
    m.b = bh / p.nv;
    m.hu = ui - m.b * p.nv * USL;
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

// Queue the operands of tokens [cb, cb + tc) of the unit's row.
template <typename ST, int K>
__device__ __forceinline__ void short_issue_tokens(const StepParams &p, const ShortMeta &m, int cb, int tc,
                                                   uint4 *stage) {
    using W = WinShape<ST, K>;
    using P = ShortTile<ST, K>;
    constexpr int RQ = K / 4;  // raw chunks per q / k vector
    constexpr int RV = 2 * RQ + W::TV;
    const int h = m.hu / P::USL, us = m.hu % P::USL;
    const int hk = h / p.r;
    uint4 *tok = stage + P::S_STATE;
    for (int ch = threadIdx.x; ch < tc * RV; ch += W::NT) {
        const int tt = ch / RV, r = ch - tt * RV;
        const float *trow = p.qkv + (long long)(m.t0 + cb + tt) * p.qkv_ss;
        const float *g;
        int dst;
        if (r < RQ) {
            g = trow + hk * K + 4 * r;
            dst = tpos<ST, K>(4 * r) / 4;
        } else if (r < 2 * RQ) {
            g = trow + (p.nk + hk) * K + 4 * (r - RQ);
            dst = W::TQ + tpos<ST, K>(4 * (r - RQ)) / 4;
        } else {
            g = trow + 2 * p.nk * K + h * K + us * P::CW + 4 * (r - 2 * RQ);
            dst = 2 * W::TQ + (r - 2 * RQ);
        }
        cp_async16(tok + tt * W::TOK + dst, g);
    }
    for (int tt = threadIdx.x; tt < tc; tt += W::NT) {
        float *ab = reinterpret_cast<float *>(tok + tt * W::TOK + W::TOKV);
        const long long o = (long long)(m.t0 + cb + tt) * p.tok_ss + (long long)h * p.tok_hs;
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
        const int h = m.hu / P::USL, us = m.hu % P::USL;
        tile_issue<ST, K, W::NT, kShortWarps>(reinterpret_cast<const ST *>(p.state) + (long long)m.slot * p.st_slot +
                                     (long long)h * p.st_head + us * P::CW,
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
    return reinterpret_cast<ST *>(tile + r * P::CPR + ((col / EPC) ^ ((r >> 3) & (P::CPR - 1)))) + (col % EPC);
}

// Writes the float32 state s (this lane's ROWS rows x C columns) into the tile.
template <typename ST, int K>
__device__ __forceinline__ void short_put_tile(uint4 *tile, int r0, int col,
                                               const float (&s)[WinShape<ST, K>::ROWS][WinShape<ST, K>::C]) {
    constexpr int ROWS = WinShape<ST, K>::ROWS, C = WinShape<ST, K>::C;
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
        Pack<ST, C> x;
#pragma unroll
        for (int c = 0; c < C; ++c) x.set(c, s[i][c]);
        x.store(tile_cols<ST, K>(tile, r0 + i, col));
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
    constexpr int V = K, NG = K / 8, LK = W::LK, RG = W::RG, ROWS = W::ROWS, C = W::C, NW = W::NW;
    constexpr int TCH = W::TCH;
    // Across few lanes a butterfly (every lane ends with every sum, two shuffle
    // rounds for LK = 4) has a shorter critical path than reduce-scatter +
    // broadcast; both follow the same tree.
    constexpr bool kUseRS = LK == 2 * C && LK > 4;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kl = lane % LK, vl = lane / LK;
    const int h = m.hu / P::USL, us = m.hu % P::USL;
    const int jr = h % p.r;
    const bool leader = tid == 0 && m.hu == 0;
    if (m.t0 < 0 || m.t1 < m.t0 || m.t1 > p.T) {
        if (leader) flag(p.status, GDR_STATUS_BAD_OFFSETS);
        return false;
    }
    const int L = m.t1 - m.t0;
    if (L == 0) return false;
    if (max_len > 0 && L > max_len) {
        if (leader) flag(p.status, GDR_STATUS_ROW_TOO_LONG);
        return false;
    }
    const int col = warp * W::WC + vl * C;  // inside the unit's tile
    float *obase = p.out + (long long)m.t0 * p.out_ss + (long long)(h * V + us * P::CW + col) * p.out_vs;
    if (m.slot < 0 || m.slot >= p.max_slots) {
        if (m.slot != -1 && leader) flag(p.status, GDR_STATUS_BAD_SLOT);
        if (kl == 0) {
            float z[C];
#pragma unroll
            for (int c = 0; c < C; ++c) z[c] = 0.0f;
            for (int t = 0; t < L; ++t) store_f32<C>(obase + (long long)t * p.out_ss, p.out_vs, p.out_vec, z);
        }
        return false;
    }
    // Verify: rows of at most ring_len tokens record and leave the pool alone.
    bool records = false, commit = true;
    float *ring_row = nullptr;
    if constexpr (MODE == Mode::Verify) {
        if (L <= rp.len) {
            commit = false;
            const int rs = rp.ring_slot[m.b];
            if (rs < 0 || rs >= rp.rows) {
                if (leader) flag(p.status, GDR_STATUS_BAD_RING_SLOT);
            } else {
                records = true;
                ring_row = rp.ring + ((long long)rs * p.nk + h / p.r) * rp.len * rp.stride;
            }
        }
    }

    const int r0 = kl * ROWS;  // this lane's first tile row
    float s[ROWS][C];
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
        Pack<ST, C> x;
        x.load(tile_cols<ST, K>(stage, r0 + i, col));
#pragma unroll
        for (int c = 0; c < C; ++c) s[i][c] = x.get(c);
    }
    float *tokf = reinterpret_cast<float *>(stage + P::S_STATE);
    bool overflow = false;
    // Per-lane output and record pointers, advanced by one token per step.
    // With the reduce-scatter the lane pair (kl, kl^1) owns column ocol; the
    // even lane writes it.  Otherwise lanes kl == 0 write all C columns.
    int ocol = col;
    bool w_out = kl == 0;
    if constexpr (kUseRS) {
        ocol = col + rs_column<LK, C>(kl);
        w_out = !(kl & 1);
    }
    float *optr = p.out + (long long)m.t0 * p.out_ss + (long long)(h * V + us * P::CW + ocol) * p.out_vs;
    float *uptr0 = ring_row;  // record of the current token
    float *uptr = records ? ring_row + rp.u_off + jr * V + us * P::CW + ocol : nullptr;
    const bool w_alpha = records && us == 0 && tid == 0;
    const bool w_kh = records && us == 0 && jr == 0 && warp == 0 && vl == 0;

    for (int cb = 0; cb < L; cb += TCH) {
        const int tc = min(TCH, L - cb);
        if (cb > 0) {  // a longer row: bring in its next chunk of operands
            __syncthreads();
            short_issue_tokens<ST, K>(p, m, cb, tc, stage);
            cp_async_commit();
            cp_async_wait<0>();
            __syncthreads();
        }
        // normalise: warp w takes tokens w, w+NW, ...; lane l works on row group l % NG
        for (int tt = warp; tt < tc; tt += NW) {
            float *tq = tokf + tt * W::TOK * 4;
            float *tk = tq + W::KP;
            float *ab = tq + W::TOKV * 4;
            const int g = lane % NG;
            const int o = tpos<ST, K>(g * 8);
            float q8[8], k8[8];
#pragma unroll
            for (int i = 0; i < 8; i += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(tq + o + i);
                const float4 b4 = *reinterpret_cast<const float4 *>(tk + o + i);
                q8[i] = a4.x; q8[i + 1] = a4.y; q8[i + 2] = a4.z; q8[i + 3] = a4.w;
                k8[i] = b4.x; k8[i + 1] = b4.y; k8[i + 2] = b4.z; k8[i + 3] = b4.w;
            }
            float ssq = chain_first(q8[0], q8[0]), ssk = chain_first(k8[0], k8[0]);
            float kqr = chain_first(k8[0], q8[0]);
#pragma unroll
            for (int i = 1; i < 8; ++i) {
                ssq = chain_next(q8[i], q8[i], ssq);
                ssk = chain_next(k8[i], k8[i], ssk);
                kqr = chain_next(k8[i], q8[i], kqr);
            }
            ssq = tree_lanes<NG>(ssq);
            ssk = tree_lanes<NG>(ssk);
            kqr = tree_lanes<NG>(kqr);
            float inv_k, qsc, kq;
            gdr_norm_scalars(ssq, ssk, kqr, p.l2norm, p.scale, p.eps, inv_k, qsc, kq);
            const float alpha = gdr_alpha(ab[0], p.decay_is_log);
            __syncwarp();
            if (lane < NG) {
#pragma unroll
                for (int i = 0; i < 8; i += 4) {
                    *reinterpret_cast<float4 *>(tk + o + i) =
                        make_float4(__fmul_rn(k8[i], inv_k), __fmul_rn(k8[i + 1], inv_k),
                                    __fmul_rn(k8[i + 2], inv_k), __fmul_rn(k8[i + 3], inv_k));
                    *reinterpret_cast<float4 *>(tq + o + i) =
                        make_float4(__fmul_rn(q8[i], qsc), __fmul_rn(q8[i + 1], qsc),
                                    __fmul_rn(q8[i + 2], qsc), __fmul_rn(q8[i + 3], qsc));
                }
            }
            if (lane == 0) {
                ab[0] = alpha;
                ab[2] = kq;
            }
        }
        __syncthreads();

        const float *tq = tokf;  // operands of token cb + tt, advanced per token
        for (int tt = 0; tt < tc; ++tt, tq += W::TOK * 4) {
            const float *tk = tq + W::KP;
            const float *ab = tq + W::TOKV * 4;
            const float alpha = ab[0], beta = ab[1], kq = ab[2];
            const int base = tpos<ST, K>(r0);  // this lane's run of rows in the staged vectors
            // a = S^T k^, b = S^T q~: one chain per 8-row group, then the tree.
            float pa[RG][C], pb[RG][C];
#pragma unroll
            for (int g = 0; g < RG; ++g) {
                float kh[8], qt[8];
#pragma unroll
                for (int i = 0; i < 8; i += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(tk + base + g * 8 + i);
                    const float4 b4 = *reinterpret_cast<const float4 *>(tq + base + g * 8 + i);
                    kh[i] = a4.x; kh[i + 1] = a4.y; kh[i + 2] = a4.z; kh[i + 3] = a4.w;
                    qt[i] = b4.x; qt[i + 1] = b4.y; qt[i + 2] = b4.z; qt[i + 3] = b4.w;
                }
                chain_first_cols<C>(s[g * 8], kh[0], pa[g]);
                chain_first_cols<C>(s[g * 8], qt[0], pb[g]);
#pragma unroll
                for (int i = 1; i < 8; ++i) {
                    chain_next_cols<C>(s[g * 8 + i], kh[i], pa[g]);
                    chain_next_cols<C>(s[g * 8 + i], qt[i], pb[g]);
                }
            }
            float a[C], bq[C];
#pragma unroll
            for (int c = 0; c < C; ++c) {
                float ac[RG], bc[RG];
#pragma unroll
                for (int g = 0; g < RG; ++g) {
                    ac[g] = pa[g][c];
                    bc[g] = pb[g][c];
                }
                a[c] = tree<RG>(ac);
                bq[c] = tree<RG>(bc);
            }
            const float *tv = tq + 2 * W::KP;
            float u[C];
            if constexpr (kUseRS) {
                float A, B;
                rs_reduce<LK, C>(a, bq, kl, A, B);
                const float uc = gdr_u(beta, alpha, A, tv[ocol]);
                if (w_out) {
                    *optr = gdr_o(alpha, B, kq, uc);
                    if (records) *uptr = uc;
                }
                rs_broadcast<LK, C>(uc, lane, u);
            } else {
#pragma unroll
                for (int c = 0; c < C; ++c) {
                    const float A = tree_lanes<LK>(a[c]);
                    const float B = tree_lanes<LK>(bq[c]);
                    u[c] = gdr_u(beta, alpha, A, tv[col + c]);
                    a[c] = gdr_o(alpha, B, kq, u[c]);  // the output
                }
                if (w_out) {
                    store_f32<C>(optr, p.out_vs, p.out_vec, a);
                    if (records) {
#pragma unroll
                        for (int c = 0; c < C; ++c) uptr[c] = u[c];
                    }
                }
            }
            if (w_alpha) uptr0[rp.alpha_off + jr] = alpha;
            if (w_kh) {
#pragma unroll
                for (int i = 0; i < ROWS; i += 4)
                    *reinterpret_cast<float4 *>(uptr0 + r0 + i) = *reinterpret_cast<const float4 *>(tk + base + i);
            }
            optr += p.out_ss;
            if (records) {
                uptr += rp.stride;
                uptr0 += rp.stride;
            }
            // S <- k^ u^T + alpha S
#pragma unroll
            for (int g = 0; g < RG; ++g) {
                float kh[8];
#pragma unroll
                for (int i = 0; i < 8; i += 4) {
                    const float4 a4 = *reinterpret_cast<const float4 *>(tk + base + g * 8 + i);
                    kh[i] = a4.x; kh[i + 1] = a4.y; kh[i + 2] = a4.z; kh[i + 3] = a4.w;
                }
#pragma unroll
                for (int i = 0; i < 8; ++i) advance_cols<C>(s[g * 8 + i], kh[i], u, alpha);
            }
            const int step = cb + tt;  // token index inside the row
            if constexpr (MODE == Mode::Snap) {
                if ((step + 1) % sp.spt == 0) {
                    const int i = (step + 1) / sp.spt - 1;
                    if (i < sp.n_inter) {
                        short_put_tile<ST, K>(stage, r0, col, s);
                        __syncthreads();
                        tile_store<ST, K, W::NT, kShortWarps>(reinterpret_cast<ST *>(sp.inter) + (long long)m.slot * sp.s_slot +
                                                     (long long)i * sp.s_tok + (long long)h * sp.s_head +
                                                     us * P::CW,
                                                 V, stage);
                        __syncthreads();
                    } else {
                        overflow = true;
                    }
                }
            }
        }
    }
    if constexpr (MODE == Mode::Snap) {
        if (overflow && leader) flag(p.status, GDR_STATUS_SNAPSHOT_OVERFLOW);
    }
    if (commit) short_put_tile<ST, K>(stage, r0, col, s);
    return commit;
}

template <typename ST, int K, Mode MODE>
__global__ void __launch_bounds__(WinShape<ST, K>::NT, kShortMinBlocks)
    k_short(const StepParams p, const RingParams rp, const SnapParams sp, const long long max_len,
            const int nunits) {
    using P = ShortTile<ST, K>;
    using W = WinShape<ST, K>;
    extern __shared__ uint4 smem_short[];
    uint4 *stage0 = smem_short, *stage1 = smem_short + W::SC;
    const long long G = gridDim.x;
    ShortMeta cur = short_meta<P::USL>(p, blockIdx.x, nunits);
    short_issue<ST, K>(p, cur, max_len, stage0);
    ShortMeta nxt = short_meta<P::USL>(p, (long long)blockIdx.x + G, nunits);
    int sel = 0;
    for (long long u = blockIdx.x; u < nunits; u += G) {
        uint4 *s_cur = sel ? stage1 : stage0;
        uint4 *s_nxt = sel ? stage0 : stage1;
        short_issue<ST, K>(p, nxt, max_len, s_nxt);
        const ShortMeta later = short_meta<P::USL>(p, u + 2 * G, nunits);
        cp_async_wait<1>();
        __syncthreads();
        const bool commit = short_compute<ST, K, MODE>(p, rp, sp, max_len, cur, s_cur);
        __syncthreads();
        if (commit) {
            const int h = cur.hu / P::USL, us = cur.hu % P::USL;
            tile_store<ST, K, W::NT, kShortWarps>(reinterpret_cast<ST *>(p.state) + (long long)cur.slot * p.st_slot +
                                         (long long)h * p.st_head + us * P::CW,
                                     p.st_k, s_cur);
        }
        __syncthreads();
        cur = nxt;
        nxt = later;
        sel ^= 1;
    }
    cp_async_wait<0>();
}

template <typename ST, int K, Mode MODE>
static cudaError_t launch_short_m(const StepParams &p, const RingParams &rp, const SnapParams &sp,
                                  long long max_len, cudaStream_t st) {
    using P = ShortTile<ST, K>;
    using W = WinShape<ST, K>;
    constexpr int SMEM = 2 * W::SMEM1;
    static int configured[64] = {0};
    static int sms[64] = {0}, occ[64] = {0};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    if (!configured[dev]) {
        e = cudaFuncSetAttribute(k_short<ST, K, MODE>, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM);
        if (e != cudaSuccess) return e;
        e = cudaDeviceGetAttribute(&sms[dev], cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[dev], k_short<ST, K, MODE>, W::NT, SMEM);
        if (e != cudaSuccess) return e;
        if (occ[dev] < 1) occ[dev] = 1;
        configured[dev] = 1;
    }
    const long long nunits = (long long)p.batch * p.nv * P::USL;
    long long grid = (long long)sms[dev] * occ[dev];
    if (grid > nunits) grid = nunits;
    if (grid > 0) k_short<ST, K, MODE><<<(unsigned)grid, W::NT, SMEM, st>>>(p, rp, sp, max_len, (int)nunits);
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
            case Mode::Snap: return launch_short_m<ST, K, Mode::Snap>(p, rp, sp, max_len, st);
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
