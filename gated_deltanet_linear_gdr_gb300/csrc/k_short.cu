// Short-row pipelined kernel: forward, verify-ring and snapshot passes over
// rows of a few tokens -- speculative-decoding verify windows
// ("gated_delta_recurrence_verify_ring_gpu") and Gated Delta Product draft
// sequences ("core.ssm.ops.gdp.fused_recurrent", intermediate_states).
//
// Persistent CTAs walk (row, value head, CW-column tile) units like the
// pipelined decode kernel.  A unit's stage holds the bf16/f32 state tile and
// the operands of its first TCH tokens, all copied with cp.async while the
// previous unit computes.  The tile is widened into float32 registers once
// (lane = 8 rows x C columns) and stays there for the whole row.  For each
// staged chunk the CTA's warps first normalise one token each (q~, k^, alpha
// and k^.q~ written back into the stage), then every warp runs the chunk's
// tokens on its columns with warp shuffles only.  Snapshots and the final
// commit go back through the stage and leave the SM as coalesced rows.  Rows
// longer than TCH load further chunks in place.  The arithmetic is the fixed
// sequence of gdr_device.cuh, so results equal the other kernels' bit for bit.
#include "gdr_pipe.cuh"

namespace gdr {

template <typename ST, int K> struct ShortShape {
    using P = PipeShape<ST, K>;
    static constexpr int TCH = 8;                        // tokens per staged chunk
    static constexpr int TQ = K / 4, TK = K / 4, TV = P::CW / 4;
    static constexpr int TOKV = TQ + TK + TV;            // 16-byte vector chunks per token
    static constexpr int TOK = TOKV + 1;                 // + {decay -> alpha, beta, k^.q~, -}
    static constexpr int SC = P::S_STATE + TCH * TOK;    // chunks per stage
    static constexpr int SMEM1 = SC * 16;
};

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
    using Sh = ShortShape<ST, K>;
    using P = PipeShape<ST, K>;
    const int h = m.hu / P::USL, us = m.hu % P::USL;
    const int hk = h / p.r;
    uint4 *tok = stage + P::S_STATE;
    for (int ch = threadIdx.x; ch < tc * Sh::TOKV; ch += P::NT) {
        const int tt = ch / Sh::TOKV, r = ch - tt * Sh::TOKV;
        const float *trow = p.qkv + (long long)(m.t0 + cb + tt) * p.qkv_ss;
        const float *g = r < Sh::TQ ? trow + hk * K + 4 * r
                         : r < Sh::TQ + Sh::TK ? trow + (p.nk + hk) * K + 4 * (r - Sh::TQ)
                                               : trow + 2 * p.nk * K + h * K + us * P::CW +
                                                     4 * (r - Sh::TQ - Sh::TK);
        cp_async16(tok + tt * Sh::TOK + r, g);
    }
    for (int tt = threadIdx.x; tt < tc; tt += P::NT) {
        float *ab = reinterpret_cast<float *>(tok + tt * Sh::TOK + Sh::TOKV);
        const long long o = (long long)(m.t0 + cb + tt) * p.tok_ss + (long long)h * p.tok_hs;
        cp_async4(ab, p.decay + o);
        cp_async4(ab + 1, p.beta + o);
    }
}

template <typename ST, int K>
__device__ __forceinline__ void short_issue(const StepParams &p, const ShortMeta &m, long long max_len,
                                            uint4 *stage) {
    using P = PipeShape<ST, K>;
    constexpr int TCH = ShortShape<ST, K>::TCH;
    if (short_unit_valid(p, m, max_len)) {
        const int h = m.hu / P::USL, us = m.hu % P::USL;
        tile_issue<ST, K>(reinterpret_cast<const ST *>(p.state) + (long long)m.slot * p.st_slot +
                              (long long)h * p.st_head + us * P::CW,
                          p.st_k, stage);
        const int L = m.t1 - m.t0;
        short_issue_tokens<ST, K>(p, m, 0, L < TCH ? L : TCH, stage);
    }
    cp_async_commit();
}

// Writes the float32 state s (this lane's 8 rows x C columns) into the tile.
template <typename ST, int K>
__device__ __forceinline__ void short_put_tile(uint4 *mine, const float (&s)[8][PipeShape<ST, K>::C]) {
    constexpr int C = PipeShape<ST, K>::C, CPR = PipeShape<ST, K>::CPR;
#pragma unroll
    for (int i = 0; i < 8; ++i) pack_store<ST, C>(mine + i * CPR, s[i]);
}

// Computes one unit; returns true when the state must be committed (the new
// tile is then in the stage, to be stored by the caller after a barrier).
// Every branch that decides between barriers is uniform over the CTA.
template <typename ST, int K, Mode MODE>
__device__ __forceinline__ bool short_compute(const StepParams &p, const RingParams &rp, const SnapParams &sp,
                                              long long max_len, const ShortMeta &m, uint4 *stage) {
    using P = PipeShape<ST, K>;
    using Sh = ShortShape<ST, K>;
    constexpr int V = K, NG = K / 8, LK = P::LK, C = P::C, CPR = P::CPR, NW = P::NW, TCH = Sh::TCH;
    using VT = typename Pack<ST, C>::VT;
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
    const int col = warp * P::WC + vl * C;  // inside the unit's tile
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

    uint4 *mine = tile_lane_base<ST, K>(stage, kl, col);
    float s[8][C];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        Pack<ST, C> x;
        x.u.v = *reinterpret_cast<const VT *>(mine + i * CPR);
#pragma unroll
        for (int c = 0; c < C; ++c) s[i][c] = x.get(c);
    }
    float *tokf = reinterpret_cast<float *>(stage + P::S_STATE);
    bool overflow = false;

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
            float *tq = tokf + tt * Sh::TOK * 4;
            float *tk = tq + K;
            float *ab = tq + Sh::TOKV * 4;
            const int g = lane % NG;
            float q8[8], k8[8];
#pragma unroll
            for (int i = 0; i < 8; i += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(tq + g * 8 + i);
                const float4 b4 = *reinterpret_cast<const float4 *>(tk + g * 8 + i);
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
                    *reinterpret_cast<float4 *>(tk + g * 8 + i) =
                        make_float4(__fmul_rn(k8[i], inv_k), __fmul_rn(k8[i + 1], inv_k),
                                    __fmul_rn(k8[i + 2], inv_k), __fmul_rn(k8[i + 3], inv_k));
                    *reinterpret_cast<float4 *>(tq + g * 8 + i) =
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

        for (int tt = 0; tt < tc; ++tt) {
            const float *tq = tokf + tt * Sh::TOK * 4;
            const float *tk = tq + K;
            const float *tv = tk + K;
            const float *ab = tq + Sh::TOKV * 4;
            const float alpha = ab[0], beta = ab[1], kq = ab[2];
            float kh[8], qt[8];
#pragma unroll
            for (int i = 0; i < 8; i += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(tk + kl * 8 + i);
                const float4 b4 = *reinterpret_cast<const float4 *>(tq + kl * 8 + i);
                kh[i] = a4.x; kh[i + 1] = a4.y; kh[i + 2] = a4.z; kh[i + 3] = a4.w;
                qt[i] = b4.x; qt[i + 1] = b4.y; qt[i + 2] = b4.z; qt[i + 3] = b4.w;
            }
            float a[C], bq[C];
            chain_first_cols<C>(s[0], kh[0], a);
            chain_first_cols<C>(s[0], qt[0], bq);
#pragma unroll
            for (int i = 1; i < 8; ++i) {
                chain_next_cols<C>(s[i], kh[i], a);
                chain_next_cols<C>(s[i], qt[i], bq);
            }
            const int step = cb + tt;  // token index inside the row
            float *orow = obase + (long long)step * p.out_ss;
            float *rec = records ? ring_row + (long long)step * rp.stride : nullptr;
            float u[C];
            if constexpr (LK == 2 * C) {
                float A, B;
                rs_reduce<LK, C>(a, bq, kl, A, B);
                const int c = rs_column<LK, C>(kl);
                const float uc = gdr_u(beta, alpha, A, tv[col + c]);
                if (!(kl & 1)) {
                    orow[(long long)c * p.out_vs] = gdr_o(alpha, B, kq, uc);
                    if (records) rec[rp.u_off + jr * V + us * P::CW + col + c] = uc;
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
                if (kl == 0) {
                    store_f32<C>(orow, p.out_vs, p.out_vec, a);
                    if (records) {
#pragma unroll
                        for (int c = 0; c < C; ++c) rec[rp.u_off + jr * V + us * P::CW + col + c] = u[c];
                    }
                }
            }
            if (records && us == 0) {
                if (tid == 0) rec[rp.alpha_off + jr] = alpha;
                if (jr == 0 && warp == 0 && vl == 0) {
                    *reinterpret_cast<float4 *>(rec + kl * 8) = make_float4(kh[0], kh[1], kh[2], kh[3]);
                    *reinterpret_cast<float4 *>(rec + kl * 8 + 4) = make_float4(kh[4], kh[5], kh[6], kh[7]);
                }
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) advance_cols<C>(s[i], kh[i], u, alpha);
            if constexpr (MODE == Mode::Snap) {
                if ((step + 1) % sp.spt == 0) {
                    const int i = (step + 1) / sp.spt - 1;
                    if (i < sp.n_inter) {
                        short_put_tile<ST, K>(mine, s);
                        __syncthreads();
                        tile_store<ST, K>(reinterpret_cast<ST *>(sp.inter) + (long long)m.slot * sp.s_slot +
                                              (long long)i * sp.s_tok + (long long)h * sp.s_head + us * P::CW,
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
    if (commit) short_put_tile<ST, K>(mine, s);
    return commit;
}

template <typename ST, int K, Mode MODE>
__global__ void __launch_bounds__(PipeShape<ST, K>::NT, 2)
    k_short(const StepParams p, const RingParams rp, const SnapParams sp, const long long max_len,
            const int nunits) {
    using P = PipeShape<ST, K>;
    using Sh = ShortShape<ST, K>;
    extern __shared__ uint4 smem_short[];
    uint4 *stage0 = smem_short, *stage1 = smem_short + Sh::SC;
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
            tile_store<ST, K>(reinterpret_cast<ST *>(p.state) + (long long)cur.slot * p.st_slot +
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
    using P = PipeShape<ST, K>;
    constexpr int SMEM = 2 * ShortShape<ST, K>::SMEM1;
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
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ[dev], k_short<ST, K, MODE>, P::NT, SMEM);
        if (e != cudaSuccess) return e;
        if (occ[dev] < 1) occ[dev] = 1;
        configured[dev] = 1;
    }
    const long long nunits = (long long)p.batch * p.nv * P::USL;
    long long grid = (long long)sms[dev] * occ[dev];
    if (grid > nunits) grid = nunits;
    if (grid > 0) k_short<ST, K, MODE><<<(unsigned)grid, P::NT, SMEM, st>>>(p, rp, sp, max_len, (int)nunits);
    return cudaGetLastError();
}

template <typename ST, int K>
static bool short_ok(const StepParams &p) {
    if constexpr (!PipeShape<ST, K>::OK) {
        return false;
    } else {
        return p.qkv_vec && (long long)p.batch * p.nv * PipeShape<ST, K>::USL < (1ll << 31);
    }
}

template <typename ST, int K>
static cudaError_t launch_short_t(const StepParams &p, Mode mode, const RingParams &rp, const SnapParams &sp,
                                  long long max_len, cudaStream_t st, bool *used) {
    *used = short_ok<ST, K>(p);
    if (!*used) return cudaSuccess;
    if constexpr (PipeShape<ST, K>::OK) {
        switch (mode) {
            case Mode::Fwd: return launch_short_m<ST, K, Mode::Fwd>(p, rp, sp, max_len, st);
            case Mode::Verify: return launch_short_m<ST, K, Mode::Verify>(p, rp, sp, max_len, st);
            case Mode::Snap: return launch_short_m<ST, K, Mode::Snap>(p, rp, sp, max_len, st);
        }
    }
    return cudaErrorInvalidValue;
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
