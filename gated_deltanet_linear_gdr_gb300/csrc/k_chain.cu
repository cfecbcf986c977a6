// General multi-token kernel: forward, verify-ring and snapshot passes.
//
// A CTA owns one (row, value head, slice of VS value columns) for the whole
// row and keeps its K x VS piece of the state in registers in float32
// ("gated_delta_recurrence_fwd_gpu" summary: the state stays in registers for
// the whole sequence).  Each warp owns 16 of the columns and all K rows:
// lane kl = lane % LK holds RG consecutive row groups (8*RG rows), lane
// vl = lane / LK holds C columns.  The K-reductions of a token therefore end
// with log2(LK) xor-shuffles and the warps never wait for each other inside a
// token.
//
// Per-token operands (raw q and k of the key head, v of the slice, alpha,
// beta) are staged in shared memory TC tokens at a time; the CTA's warps then
// normalise the staged q, k once per token (shared by all warps) and run the
// TC tokens.  One sweep over the state per token applies the update of token
// t and accumulates the reductions of token t+1 (the readout identity in
// gdr_device.cuh makes both reductions act on the pre-decay state).
#include "gdr_device.cuh"

namespace gdr {

template <typename ST, int K> struct ChainShape {
    static constexpr int V = K;
    static constexpr int NG = K / 8;               // row groups
    static constexpr int LK = cmin(4, NG);         // lanes along K
    static constexpr int RG = NG / LK;             // groups per lane
    static constexpr int ROWS = RG * 8;            // rows per lane
    static constexpr int LV = 32 / LK;             // lanes along V
    static constexpr int C = cmin(2, V / LV);      // columns per lane
    static constexpr int WC = LV * C;              // columns per warp (16)
    static constexpr int W = cmin(4, V / WC);      // warps per CTA
    static constexpr int NT = 32 * W;
    static constexpr int VS = W * WC;              // columns per CTA
    static constexpr int SLICES = V / VS;
    static constexpr int KP = K + LK * 4;          // padded staged vector length
    static constexpr int TC = 16;                  // tokens per staged chunk
};

// Padded shared-memory index of row i: 4 spare floats after each lane's run of
// rows keeps the LK distinct 16-byte reads of one warp instruction in
// different banks.
template <int ROWS> __device__ __forceinline__ int pidx(int i) { return i + (i / ROWS) * 4; }

template <typename ST, int K, Mode MODE>
__global__ void __launch_bounds__(ChainShape<ST, K>::NT)
    k_chain(const StepParams p, const RingParams rp, const SnapParams sp, const long long max_len) {
    using Sh = ChainShape<ST, K>;
    constexpr int V = K, NG = Sh::NG, LK = Sh::LK, RG = Sh::RG, ROWS = Sh::ROWS, C = Sh::C;
    constexpr int WC = Sh::WC, W = Sh::W, NT = Sh::NT, VS = Sh::VS, SLICES = Sh::SLICES;
    constexpr int KP = Sh::KP, TC = Sh::TC;

    // two chunk buffers: chunk i+1 is copied in while chunk i is processed
    __shared__ __align__(16) float q_s[2][TC][KP];
    __shared__ __align__(16) float k_s[2][TC][KP];
    __shared__ __align__(16) float v_s[2][TC][VS];
    __shared__ __align__(16) float sc_s[2][TC][4];  // decay -> alpha, beta, k^.q~

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kl = lane % LK, vl = lane / LK;
    const int slice = (int)(blockIdx.x % SLICES);
    const long long bh = blockIdx.x / SLICES;
    const int h = (int)(bh % p.nv);
    const int b = (int)(bh / p.nv);
    const bool leader = tid == 0 && slice == 0 && h == 0;

    const int t0 = p.offsets[b], t1 = p.offsets[b + 1];
    if (t0 < 0 || t1 < t0 || t1 > p.T) {
        if (leader) flag(p.status, GDR_STATUS_BAD_OFFSETS);
        return;
    }
    const int L = t1 - t0;
    if (L == 0) return;
    if (max_len > 0 && L > max_len) {
        if (leader) flag(p.status, GDR_STATUS_ROW_TOO_LONG);
        return;
    }
    const int wcol = warp * WC + vl * C;           // lane's first column inside the slice
    const int col0 = slice * VS + wcol;            // ... inside the head
    float *obase = p.out + (long long)t0 * p.out_ss + (long long)(h * V + col0) * p.out_vs;
    const int slot = p.slot_idx[b];
    if (slot < 0 || slot >= p.max_slots) {
        if (slot != -1 && leader) flag(p.status, GDR_STATUS_BAD_SLOT);
        if (kl == 0) {
            float z[C];
#pragma unroll
            for (int c = 0; c < C; ++c) z[c] = 0.0f;
            for (int t = 0; t < L; ++t) store_f32<C>(obase + (long long)t * p.out_ss, p.out_vs, p.out_vec, z);
        }
        return;
    }

    // Verify: rows of at most ring_len tokens record; longer rows commit.
    bool records = false, commit = true;
    float *ring_row = nullptr;
    const int hk = h / p.r, jr = h % p.r;
    if constexpr (MODE == Mode::Verify) {
        if (L <= rp.len) {
            commit = false;
            const int rs = rp.ring_slot[b];
            if (rs < 0 || rs >= rp.rows) {
                if (leader) flag(p.status, GDR_STATUS_BAD_RING_SLOT);
            } else {
                records = true;
                ring_row = rp.ring + ((long long)rs * p.nk + hk) * rp.len * rp.stride;
            }
        }
    }

    // State piece: rows kl*ROWS .. +ROWS, columns col0 .. col0+C.
    ST *stile = reinterpret_cast<ST *>(p.state) + (long long)slot * p.st_slot +
                (long long)h * p.st_head + (long long)(kl * ROWS) * p.st_k + col0;
    float s[ROWS][C];
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
        Pack<ST, C> x;
        x.load(stile + i * p.st_k);
#pragma unroll
        for (int c = 0; c < C; ++c) s[i][c] = x.get(c);
    }

    const long long qoff = (long long)(hk * K) * p.qkv_cs;
    const long long koff = (long long)(p.nk * K + hk * K) * p.qkv_cs;
    const long long voff = (long long)(2 * p.nk * K + h * V + slice * VS) * p.qkv_cs;
    bool overflow = false;

    // Raw operands of tokens [cb, cb + tc) into buffer bi; one cp.async group.
    auto stage = [&](int cb, int tc, int bi) {
        if (p.qkv_vec) {
            constexpr int RQ = K / 4, RVS = VS / 4, RT = 2 * RQ + RVS;
            for (int idx = tid; idx < tc * RT; idx += NT) {
                const int tt = idx / RT, r = idx - tt * RT;
                const float *row = p.qkv + (long long)(t0 + cb + tt) * p.qkv_ss;
                if (r < RQ)
                    cp_async16(&q_s[bi][tt][pidx<ROWS>(4 * r)], row + qoff + 4 * r);
                else if (r < 2 * RQ)
                    cp_async16(&k_s[bi][tt][pidx<ROWS>(4 * (r - RQ))], row + koff + 4 * (r - RQ));
                else
                    cp_async16(&v_s[bi][tt][4 * (r - 2 * RQ)], row + voff + 4 * (r - 2 * RQ));
            }
            for (int tt = tid; tt < tc; tt += NT) {
                const long long o = (long long)(t0 + cb + tt) * p.tok_ss + (long long)h * p.tok_hs;
                cp_async4(&sc_s[bi][tt][0], p.decay + o);
                cp_async4(&sc_s[bi][tt][1], p.beta + o);
            }
        } else {
            for (int idx = tid; idx < tc * K; idx += NT) {
                const int tt = idx / K, i = idx - tt * K;
                const float *row = p.qkv + (long long)(t0 + cb + tt) * p.qkv_ss;
                q_s[bi][tt][pidx<ROWS>(i)] = row[qoff + (long long)i * p.qkv_cs];
                k_s[bi][tt][pidx<ROWS>(i)] = row[koff + (long long)i * p.qkv_cs];
            }
            for (int idx = tid; idx < tc * VS; idx += NT) {
                const int tt = idx / VS, j = idx - tt * VS;
                v_s[bi][tt][j] = p.qkv[(long long)(t0 + cb + tt) * p.qkv_ss + voff + (long long)j * p.qkv_cs];
            }
            for (int tt = tid; tt < tc; tt += NT) {
                const long long o = (long long)(t0 + cb + tt) * p.tok_ss + (long long)h * p.tok_hs;
                sc_s[bi][tt][0] = p.decay[o];
                sc_s[bi][tt][1] = p.beta[o];
            }
        }
        cp_async_commit();
    };

    const int nch = (L + TC - 1) / TC;
    stage(0, min(TC, L), 0);
    for (int ci = 0; ci < nch; ++ci) {
        const int cb = ci * TC, tc = min(TC, L - cb), bi = ci & 1;
        if (ci + 1 < nch) {
            stage(cb + TC, min(TC, L - cb - TC), bi ^ 1);  // its buffer was released at the end of ci-1
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        float(*qb)[KP] = q_s[bi];
        float(*kb)[KP] = k_s[bi];
        float(*vb)[VS] = v_s[bi];
        float(*sb)[4] = sc_s[bi];
        // ---- normalise: warp w takes tokens w, w+W, ...; lane l works on group l % NG
        for (int tt = warp; tt < tc; tt += W) {
            const int g = lane % NG;
            const int o = pidx<ROWS>(g * 8);
            float q8[8], k8[8];
#pragma unroll
            for (int i = 0; i < 8; i += 4) {
                const float4 a4 = *reinterpret_cast<const float4 *>(&qb[tt][o + i]);
                const float4 b4 = *reinterpret_cast<const float4 *>(&kb[tt][o + i]);
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
            const float alpha = gdr_alpha(sb[tt][0], p.decay_is_log);
            __syncwarp();
            if (lane < NG) {
#pragma unroll
                for (int i = 0; i < 8; i += 4) {
                    *reinterpret_cast<float4 *>(&kb[tt][o + i]) =
                        make_float4(__fmul_rn(k8[i], inv_k), __fmul_rn(k8[i + 1], inv_k),
                                    __fmul_rn(k8[i + 2], inv_k), __fmul_rn(k8[i + 3], inv_k));
                    *reinterpret_cast<float4 *>(&qb[tt][o + i]) =
                        make_float4(__fmul_rn(q8[i], qsc), __fmul_rn(q8[i + 1], qsc),
                                    __fmul_rn(q8[i + 2], qsc), __fmul_rn(q8[i + 3], qsc));
                }
            }
            if (lane == 0) {
                sb[tt][0] = alpha;
                sb[tt][2] = kq;
            }
        }
        __syncthreads();

        // ---- reductions of the chunk's first token
        const int rb = pidx<ROWS>(kl * ROWS);  // start of this lane's rows in the staged vectors
        float pa[RG][C], pb[RG][C];
#pragma unroll
        for (int g = 0; g < RG; ++g) {
#pragma unroll
            for (int i4 = 0; i4 < 2; ++i4) {
                const float4 kn = *reinterpret_cast<const float4 *>(&kb[0][rb + g * 8 + i4 * 4]);
                const float4 qn = *reinterpret_cast<const float4 *>(&qb[0][rb + g * 8 + i4 * 4]);
                const float knv[4] = {kn.x, kn.y, kn.z, kn.w}, qnv[4] = {qn.x, qn.y, qn.z, qn.w};
#pragma unroll
                for (int ii = 0; ii < 4; ++ii) {
                    const int r = g * 8 + i4 * 4 + ii;
                    if (i4 == 0 && ii == 0) {
                        chain_first_cols<C>(s[r], knv[ii], pa[g]);
                        chain_first_cols<C>(s[r], qnv[ii], pb[g]);
                    } else {
                        chain_next_cols<C>(s[r], knv[ii], pa[g]);
                        chain_next_cols<C>(s[r], qnv[ii], pb[g]);
                    }
                }
            }
        }

        // ---- the chunk's tokens
        for (int tt = 0; tt < tc; ++tt) {
            const float alpha = sb[tt][0], beta = sb[tt][1], kq = sb[tt][2];
            float u[C], o[C];
#pragma unroll
            for (int c = 0; c < C; ++c) {
                float ac[RG], bc[RG];
#pragma unroll
                for (int g = 0; g < RG; ++g) {
                    ac[g] = pa[g][c];
                    bc[g] = pb[g][c];
                }
                const float A = tree_lanes<LK>(tree<RG>(ac));
                const float B = tree_lanes<LK>(tree<RG>(bc));
                u[c] = gdr_u(beta, alpha, A, vb[tt][wcol + c]);
                o[c] = gdr_o(alpha, B, kq, u[c]);
            }
            const int step = cb + tt;  // token index inside the row
            if (kl == 0) store_f32<C>(obase + (long long)step * p.out_ss, p.out_vs, p.out_vec, o);
            if constexpr (MODE == Mode::Verify) {
                if (records) {
                    float *rec = ring_row + (long long)step * rp.stride;
                    if (kl == 0) {
#pragma unroll
                        for (int c = 0; c < C; ++c) rec[rp.u_off + jr * V + col0 + c] = u[c];
                    }
                    if (slice == 0) {
                        if (tid == 0) rec[rp.alpha_off + jr] = alpha;
                        if (jr == 0)
                            for (int i = tid; i < K; i += NT) rec[i] = kb[tt][pidx<ROWS>(i)];
                    }
                }
            }
            // One sweep: S <- k^_t u^T + alpha S, and token t+1's partials on the new S.
            const bool next = tt + 1 < tc;
#pragma unroll
            for (int g = 0; g < RG; ++g) {
#pragma unroll
                for (int i4 = 0; i4 < 2; ++i4) {
                    const int o4 = rb + g * 8 + i4 * 4;
                    const float4 kc = *reinterpret_cast<const float4 *>(&kb[tt][o4]);
                    const float kcv[4] = {kc.x, kc.y, kc.z, kc.w};
                    float knv[4] = {0.f, 0.f, 0.f, 0.f}, qnv[4] = {0.f, 0.f, 0.f, 0.f};
                    if (next) {
                        const float4 kn = *reinterpret_cast<const float4 *>(&kb[tt + 1][o4]);
                        const float4 qn = *reinterpret_cast<const float4 *>(&qb[tt + 1][o4]);
                        knv[0] = kn.x; knv[1] = kn.y; knv[2] = kn.z; knv[3] = kn.w;
                        qnv[0] = qn.x; qnv[1] = qn.y; qnv[2] = qn.z; qnv[3] = qn.w;
                    }
#pragma unroll
                    for (int ii = 0; ii < 4; ++ii) {
                        const int r = g * 8 + i4 * 4 + ii;
                        advance_cols<C>(s[r], kcv[ii], u, alpha);
                        if (i4 == 0 && ii == 0) {
                            chain_first_cols<C>(s[r], knv[ii], pa[g]);
                            chain_first_cols<C>(s[r], qnv[ii], pb[g]);
                        } else {
                            chain_next_cols<C>(s[r], knv[ii], pa[g]);
                            chain_next_cols<C>(s[r], qnv[ii], pb[g]);
                        }
                    }
                }
            }
            if constexpr (MODE == Mode::Snap) {
                if ((step + 1) % sp.spt == 0) {
                    const int i = (step + 1) / sp.spt - 1;
                    if (i < sp.n_inter) {
                        ST *it = reinterpret_cast<ST *>(sp.inter) + (long long)slot * sp.s_slot +
                                 (long long)i * sp.s_tok + (long long)h * sp.s_head +
                                 (long long)(kl * ROWS) * V + col0;
#pragma unroll
                        for (int r = 0; r < ROWS; ++r) {
                            Pack<ST, C> x;
#pragma unroll
                            for (int c = 0; c < C; ++c) x.set(c, s[r][c]);
                            x.store(it + r * V);
                        }
                    } else {
                        overflow = true;
                    }
                }
            }
        }
        __syncthreads();  // every warp is done with buffer bi before chunk ci+2 is copied into it
    }
    if constexpr (MODE == Mode::Snap) {
        if (overflow && leader) flag(p.status, GDR_STATUS_SNAPSHOT_OVERFLOW);
    }
    (void)records;
    if (commit) {
#pragma unroll
        for (int i = 0; i < ROWS; ++i) {
            Pack<ST, C> x;
#pragma unroll
            for (int c = 0; c < C; ++c) x.set(c, s[i][c]);
            x.store(stile + i * p.st_k);
        }
    }
}

template <typename ST, int K>
static cudaError_t launch_chain_t(const StepParams &p, Mode mode, const RingParams &rp,
                                  const SnapParams &sp, long long max_len, cudaStream_t st) {
    using Sh = ChainShape<ST, K>;
    const long long blocks = (long long)p.batch * p.nv * Sh::SLICES;
    if (blocks <= 0) return cudaGetLastError();
    switch (mode) {
        case Mode::Fwd:
            k_chain<ST, K, Mode::Fwd><<<(unsigned)blocks, Sh::NT, 0, st>>>(p, rp, sp, max_len);
            break;
        case Mode::Verify:
            k_chain<ST, K, Mode::Verify><<<(unsigned)blocks, Sh::NT, 0, st>>>(p, rp, sp, max_len);
            break;
        case Mode::Snap:
            k_chain<ST, K, Mode::Snap><<<(unsigned)blocks, Sh::NT, 0, st>>>(p, rp, sp, max_len);
            break;
    }
    return cudaGetLastError();
}

cudaError_t launch_chain(const StepParams &p, int K, bool bf16, Mode mode, const RingParams &rp,
                         const SnapParams &sp, long long max_row_len, cudaStream_t s) {
#define GDR_CASE(KK)                                                                    \
    case KK:                                                                            \
        return bf16 ? launch_chain_t<uint16_t, KK>(p, mode, rp, sp, max_row_len, s)     \
                    : launch_chain_t<float, KK>(p, mode, rp, sp, max_row_len, s);
    switch (K) {
        GDR_CASE(16)
        GDR_CASE(32)
        GDR_CASE(64)
        GDR_CASE(128)
    }
#undef GDR_CASE
    return cudaErrorInvalidValue;
}

}  // namespace gdr
