// General multi-token kernel: forward, verify-ring and snapshot passes.
//
// A CTA owns one (row, value head, slice of VS value columns) for the whole
// row and keeps its K x VS piece of the state in registers in float32
// ("gated_delta_recurrence_fwd_gpu" summary: the state stays in registers for
// the whole sequence).  Each warp owns WC of the columns and all K rows:
// lane kl = lane % LK holds RG consecutive row groups (8*RG rows, in the
// row-pair form of gdr_state.cuh when RG is even), lane vl = lane / LK holds
// C columns.  The K-reductions of a token therefore end
// with log2(LK) xor-shuffles and the warps never wait for each other inside a
// token.
//
// Per-token operands (raw q and k of the key head, v of the slice, alpha,
// beta) are staged in shared memory TC tokens at a time; the CTA's warps then
// normalise the staged q, k once per token (shared by all warps) and run the
// TC tokens.  One sweep over the state per token applies the update of token
// t and accumulates the reductions of token t+1 (the readout identity in
// gdr_device.cuh makes both reductions act on the pre-decay state).
#pragma once

#include "gdr_state.cuh"

namespace gdr {

// Tokens per staged chunk TCX (8, 16 or 32, chosen by the launcher from the
// caller's row-length bound); per-element beta (BPV) stages beta per token
// like v and uses at most 8 tokens.
template <typename ST, int K, int VV = K, bool BPV = false, int TCX = 16, bool CONV = false> struct ChainShape {
    static constexpr int V = VV;                   // value head size: K, 2K or K/2
    static constexpr int NG = K / 8;               // row groups
    // lanes along K: 4 (32 rows per lane at K = 128), or 2 for K = 128 with
    // 32-token chunks or a float32 state.  Long rows run one CTA per row and
    // head for the whole row, so the work a lane carries per token sets how
    // well two CTAs per SM keep the FMA pipes busy: 64 rows per lane (a
    // whole-head CTA, 213 registers) beat 32 rows (ragged prefill 2.02 -> 1.90
    // ms) and 16 rows (2.32 ms).  Float32 snapshots gain too (154 -> 146 us:
    // each warp store covers 128 contiguous bytes of a row).  bf16 rows bounded
    // at 8 or 16 tokens keep the narrower lane, whose CTAs fit four to an SM.
    static constexpr int LK =
        (NG >= 16 && ((TCX >= 32 && !BPV) || sizeof(ST) == 4)) ? 2 : NG >= 4 ? cmin(4, NG / 2) : NG;
    static constexpr int RG = NG / LK;             // groups per lane
    static constexpr bool RPAIR = RG % 2 == 0;     // row-pair register form
    static constexpr int ROWS = RG * 8;            // rows per lane
    static constexpr int LV = 32 / LK;             // lanes along V
    static constexpr int C = cmin(2, V / LV);      // columns per lane
    static constexpr int WC = LV * C;              // columns per warp
    static constexpr int W = cmin(4, V / WC);      // warps per CTA
    static constexpr int NT = 32 * W;
    static constexpr int VS = W * WC;              // columns per CTA
    static constexpr int SLICES = V / VS;
    static constexpr int KP = K + LK * 4;          // padded staged vector length
    static constexpr int TC = BPV ? cmin(8, TCX) : TCX;  // tokens per staged chunk
    // dynamic shared memory, in floats: q, k [2][TC][KP]; v [2][TC][VS];
    // {alpha, beta, k^.q~, -} [2][TC][4]; per-element beta [2][TC][VS]
    static constexpr int SM_Q = 0, SM_K = SM_Q + 2 * TC * KP, SM_V = SM_K + 2 * TC * KP;
    static constexpr int SM_SC = SM_V + 2 * TC * VS, SM_B = SM_SC + 2 * TC * 4;
    // Pass-1 convolution (CONV): the taps (zero-filled to 4) and bias of each
    // of the CTA's channels -- its key head's q and k, its value slice --
    // [NCH][5] floats; thread tid owns channels tid, tid + NT, ... (CPT of
    // them) and keeps their last 3 raw inputs in registers
    static constexpr int NCH = 2 * K + VS;
    static constexpr int CPT = (NCH + NT - 1) / NT;
    static constexpr int SM_CV = SM_B + (BPV ? 2 * TC * VS : 0);
    static constexpr int SMEM = (SM_CV + (CONV ? NCH * 5 : 0)) * 4;  // bytes
    static constexpr int NL = NG / (RPAIR ? 2 : 1);  // lanes per token when normalising
    static constexpr int TPW = 32 / NL;            // tokens per warp when normalising
    using State = LaneState<RG, C>;
};

// Shared-memory index of raw row i (natural order, padded every ROWS rows).
template <int ROWS> __device__ __forceinline__ int pidx(int i) { return vpos<false, ROWS>(i); }

// Global channel of the CTA's convolution channel j: its key head's q (j < K),
// k (j < 2K), then its slice of value head h.
template <int K, int V, int VS>
__device__ __forceinline__ int conv_channel(int j, const StepParams &p, int hk, int h, int slice) {
    if (j < K) return hk * K + j;
    if (j < 2 * K) return p.nk * K + hk * K + (j - K);
    return 2 * p.nk * K + h * V + slice * VS + (j - 2 * K);
}

template <bool B> struct WinFull {
    static constexpr bool value = B;
};

// The causal convolution of one staged chunk of tc tokens, in place, for the
// thread's channels j = tid + i NT (Sh::CPT of them): per token and channel
// y = bias, y = fma(w[m], xe[m], y) for the WW taps m = 0 .. WW-1 over the
// window xe = (last WW-1 raw inputs, this input), then SiLU y / (1 + e^-y)
// (fast exponential and division) when asked.  Taps and bias from cv_s
// [NCH][5]; hist[i] holds channel i's last raw inputs, the newest last, and
// is carried to the next chunk.  Channel j's staged values: q for j < K, k
// for j < 2K, then the value slice.
template <typename Sh, int WW>
__device__ __forceinline__ void conv_chunk(float (*qb)[Sh::KP], float (*kb)[Sh::KP], float (*vb)[Sh::VS],
                                           const float *cv_s, float (&hist)[Sh::CPT][3], int tc, int silu) {
    constexpr int K = Sh::NG * 8, NCH = Sh::NCH, CPT = Sh::CPT, NT = Sh::NT;
    const int tid = threadIdx.x;
    float *x0[CPT];
    int xs[CPT];
    float w[CPT][4], bias[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) {
        const int j = min(tid + i * NT, NCH - 1);
        x0[i] = j < K ? &qb[0][pidx<Sh::ROWS>(j)] : j < 2 * K ? &kb[0][pidx<Sh::ROWS>(j - K)] : &vb[0][j - 2 * K];
        xs[i] = j < 2 * K ? Sh::KP : Sh::VS;
#pragma unroll
        for (int m = 0; m < 4; ++m) w[i][m] = cv_s[j * 5 + m];
        bias[i] = cv_s[j * 5 + 4];
    }
    // blocks of TB tokens: every load of a block, then its TB * CPT
    // independent outputs, then the stores (loads and stores go through
    // pointers the compiler cannot tell apart, so it would keep them in
    // order); whole blocks take a path without tail predicates
    constexpr int TB = 4;
    bool own[CPT];
#pragma unroll
    for (int i = 0; i < CPT; ++i) own[i] = tid + i * NT < NCH;
    auto block = [&](auto full, int t0) {
        constexpr bool FULL = decltype(full)::value;
        const int n = FULL ? TB : tc - t0;
        float xv[CPT][TB], yv[CPT][TB];
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            const float *px = x0[i] + t0 * xs[i];
#pragma unroll
            for (int u = 0; u < TB; ++u) xv[i][u] = own[i] && (FULL || u < n) ? px[u * xs[i]] : 0.0f;
        }
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
#pragma unroll
            for (int u = 0; u < TB; ++u) {
                // window: the WW-1 inputs before token t0+u, then its own
                float y = bias[i];
#pragma unroll
                for (int m = 0; m < WW - 1; ++m) {
                    const int back = WW - 1 - m;
                    const float xm = u - back >= 0 ? xv[i][u - back >= 0 ? u - back : 0] : hist[i][3 + u - back];
                    y = __fmaf_rn(w[i][m], xm, y);
                }
                y = __fmaf_rn(w[i][WW - 1], xv[i][u], y);
                if (silu) y = __fdividef(y, __fadd_rn(1.0f, __expf(-y)));
                yv[i][u] = y;
            }
        }
#pragma unroll
        for (int i = 0; i < CPT; ++i) {
            float *px = x0[i] + t0 * xs[i];
            if (own[i]) {
#pragma unroll
                for (int u = 0; u < TB; ++u)
                    if (FULL || u < n) px[u * xs[i]] = yv[i][u];
            }
            // history: the last three inputs up to the block's last token
            if constexpr (FULL) {
                hist[i][0] = xv[i][TB - 3];
                hist[i][1] = xv[i][TB - 2];
                hist[i][2] = xv[i][TB - 1];
            } else {
                float nh[3];
#pragma unroll
                for (int m = 0; m < 3; ++m) {
                    float v = hist[i][m];
#pragma unroll
                    for (int nn = 1; nn < TB; ++nn)
                        if (n == nn) {
                            const int pos = nn - 3 + m;  // negative: from the old history
                            v = pos >= 0 ? xv[i][pos >= 0 ? pos : 0] : hist[i][3 + pos >= 0 ? 3 + pos : 0];
                        }
                    nh[m] = v;
                }
#pragma unroll
                for (int m = 0; m < 3; ++m) hist[i][m] = nh[m];
            }
        }
    };
    int t0 = 0;
#pragma unroll 2
    for (; t0 + TB <= tc; t0 += TB) block(WinFull<true>{}, t0);
    if (t0 < tc) block(WinFull<false>{}, t0);
}

// Block -> unit for a few long rows of unequal length (every thread of the
// CTA calls it; needs blockDim.x >= batch).  A CTA owns its row for the whole
// row, so the time of the call is set by the SM whose resident CTAs hold the
// most tokens.  Units are taken in order of decreasing row length (ties by
// row index) and dealt to the blocks as a snake: pass j covers blocks
// jP .. jP+P-1 (P = SMs), forward on even passes and backward on odd ones,
// so when the first wave is spread over the SMs in a fixed order the long
// and short rows pair up on each SM.  Any placement still gets every unit
// exactly once.
__device__ __forceinline__ long long chain_balanced_unit(const StepParams &p, int slices, int P) {
    __shared__ int row_of_rank;
    const long long per_row = (long long)p.nv * slices;
    const long long n = (long long)p.batch * per_row;
    const long long i = blockIdx.x, pass = i / P, pos = i - pass * P;
    const long long m = n - pass * P < P ? n - pass * P : P;  // blocks in this pass
    const long long k = pass * P + ((pass & 1) ? m - 1 - pos : pos);
    const int rank = (int)(k / per_row);
    const int r = threadIdx.x;
    if (r < p.batch) {
        const int Lr = p.offsets[r + 1] - p.offsets[r];
        int rk = 0;
        for (int j = 0; j < p.batch; ++j) {
            const int Lj = p.offsets[j + 1] - p.offsets[j];
            rk += (Lj > Lr || (Lj == Lr && j < r)) ? 1 : 0;
        }
        if (rk == rank) row_of_rank = r;
    }
    __syncthreads();
    return (long long)row_of_rank * per_row + (k - (long long)rank * per_row);
}

// 32-token chunks take 101 KiB of shared memory at K = 128, so two CTAs fit
// an SM anyway: the register cap follows (the 64-row lane needs the extra
// registers; with 32-row lanes they already let the compiler keep more staged
// operands in flight, ragged prefill 2.10 -> 2.02 ms).  The 64-row lane takes
// the same cap with shorter chunks.
template <typename ST, int K, int VV, Mode MODE, bool BPV, int TCX, bool CONV = false>
__global__ void __launch_bounds__(ChainShape<ST, K, VV, BPV, TCX, CONV>::NT,
                                  (TCX >= 32 || ChainShape<ST, K, VV, BPV, TCX, CONV>::ROWS >= 64) ? 2 : 4)
    k_chain(const StepParams p, const RingParams rp, const SnapParams sp, const ConvParams cv, const long long max_len,
            const int order_p) {
    using Sh = ChainShape<ST, K, VV, BPV, TCX, CONV>;
    constexpr int V = VV, LK = Sh::LK, ROWS = Sh::ROWS, C = Sh::C;
    constexpr int WC = Sh::WC, W = Sh::W, NT = Sh::NT, VS = Sh::VS, SLICES = Sh::SLICES;
    constexpr int KP = Sh::KP, TC = Sh::TC, NL = Sh::NL, TPW = Sh::TPW;

    // two chunk buffers: chunk i+1 is copied in while chunk i is processed
    extern __shared__ __align__(16) float chain_smem[];
    float(*q_s)[TC][KP] = reinterpret_cast<float(*)[TC][KP]>(chain_smem + Sh::SM_Q);
    float(*k_s)[TC][KP] = reinterpret_cast<float(*)[TC][KP]>(chain_smem + Sh::SM_K);
    float(*v_s)[TC][VS] = reinterpret_cast<float(*)[TC][VS]>(chain_smem + Sh::SM_V);
    float(*sc_s)[TC][4] = reinterpret_cast<float(*)[TC][4]>(chain_smem + Sh::SM_SC);  // decay -> alpha, beta, k^.q~
    float(*b_s)[TC][VS] = reinterpret_cast<float(*)[TC][VS]>(chain_smem + Sh::SM_B);  // per-element beta

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int kl = lane % LK, vl = lane / LK;
    const long long unit = order_p > 0 ? chain_balanced_unit(p, SLICES, order_p) : (long long)blockIdx.x;
    const int slice = (int)(unit % SLICES);
    const long long bh = unit / SLICES;
    const int h = (int)(bh % p.nv);
    const int b = (int)(bh / p.nv);
    const bool leader = tid == 0 && slice == 0 && h == 0;

    const int t0 = p.offsets[b], t1 = p.offsets[b + 1];
    if (t0 < 0 || t1 < t0 || t1 > p.T) {
        if (leader) flag(p.status, GDR_STATUS_BAD_OFFSETS);
        return;
    }
    const int L = t1 - t0;
    if (L == 0 && !p.dense) return;  // the dense mode still hands the start state on
    const int wcol = warp * WC + vl * C;           // lane's first column inside the slice
    const int col0 = slice * VS + wcol;            // ... inside the head
    float *obase = p.out + (long long)t0 * p.out_ss + (long long)(h * V + col0) * p.out_vs;
    if (max_len > 0 && L > max_len) {  // longer than the caller's bound: zero output, nothing else
        if (leader) flag(p.status, GDR_STATUS_ROW_TOO_LONG);
        if (kl == 0) zero_rows<C>(obase, L, p);
        return;
    }
    const int slot = p.dense ? b : p.slot_idx[b];
    if (slot < 0 || slot >= p.max_slots) {
        if (slot != -1 && leader) flag(p.status, GDR_STATUS_BAD_SLOT);
        if (kl == 0) zero_rows<C>(obase, L, p);
        return;
    }

    // Verify: rows of at most ring_len tokens record; longer rows commit.
    bool records = false, commit = true;
    long long ring_row = 0;  // element index of this (ring row, key head)'s first record
    const int hk = h / p.r, jr = h % p.r;
    if constexpr (MODE == Mode::Verify) {
        if (L <= rp.len) {
            commit = false;
            const int rs = rp.ring_slot[b];
            if (rs < 0 || rs >= rp.rows) {
                if (leader) flag(p.status, GDR_STATUS_BAD_RING_SLOT);
            } else {
                records = true;
                ring_row = ((long long)rs * p.nk + hk) * rp.len * rp.stride;
            }
        }
    }

    // Pass-1 convolution: thread tid owns the CTA's channels j = tid + i NT
    // < NCH (q, then k, then the value slice): their taps and bias go to
    // shared memory, the slot's conv state (the last width-1 raw inputs, the
    // newest last) to the thread's history registers
    float *cv_s = chain_smem + Sh::SM_CV;  // [NCH][5]: taps 0..3, bias
    float hist[Sh::CPT][3];
    if constexpr (CONV) {
#pragma unroll
        for (int i = 0; i < Sh::CPT; ++i) {
            const int j = tid + i * NT;
            if (j < Sh::NCH) {
                const int gc = conv_channel<K, V, Sh::VS>(j, p, hk, h, slice);
#pragma unroll
                for (int m = 0; m < 4; ++m)
                    cv_s[j * 5 + m] = m < cv.width ? cv.w[(long long)gc * cv.w_cs + m * cv.w_ts] : 0.0f;
                cv_s[j * 5 + 4] = cv.bias ? cv.bias[gc] : 0.0f;
                // the width-1 stored inputs (oldest first) end at hist[i][2]
#pragma unroll
                for (int m = 0; m < 3; ++m) {
                    const int si = m - (4 - cv.width);
                    hist[i][m] = si >= 0 ? cv.state[(long long)slot * cv.cs_slot + (long long)gc * cv.cs_chan +
                                                    si * cv.cs_tap]
                                         : 0.0f;
                }
            }
        }
    }

    // State piece: rows kl*ROWS .. +ROWS, columns col0 .. col0+C, read from
    // state_in (zeros when null) and committed to state_out.
    const long long soff = (long long)slot * p.st_slot + (long long)h * p.st_head + (long long)(kl * ROWS) * p.st_k + col0;
    const ST *sin = p.state_in ? reinterpret_cast<const ST *>(p.state_in) + soff : nullptr;
    typename Sh::State s;
#pragma unroll
    for (int i = 0; i < ROWS; ++i) {
        Pack<ST, C> x;
        if (sin)
            x.load(sin + i * p.st_k);
        else
            x.u.v = {};
#pragma unroll
        for (int c = 0; c < C; ++c) s.set(i, c, x.get(c));
    }

    const long long qoff = (long long)(hk * K) * p.qkv_cs;
    const long long koff = (long long)(p.nk * K + hk * K) * p.qkv_cs;
    const long long voff = (long long)(2 * p.nk * K + h * V + slice * VS) * p.qkv_cs;
    const float *bbase = p.beta + (long long)h * p.beta_hs + (long long)(slice * VS) * p.beta_vs;  // BPV
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
                if constexpr (!BPV) cp_async4(&sc_s[bi][tt][1], p.beta + o);
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
                if constexpr (!BPV) sc_s[bi][tt][1] = p.beta[o];
            }
        }
        if constexpr (BPV) {
            if (p.beta_vec) {
                constexpr int RVS = VS / 4;
                for (int idx = tid; idx < tc * RVS; idx += NT) {
                    const int tt = idx / RVS, r = idx - tt * RVS;
                    cp_async16(&b_s[bi][tt][4 * r], bbase + (long long)(t0 + cb + tt) * p.beta_ss + 4 * r);
                }
            } else {
                for (int idx = tid; idx < tc * VS; idx += NT) {
                    const int tt = idx / VS, j = idx - tt * VS;
                    b_s[bi][tt][j] = bbase[(long long)(t0 + cb + tt) * p.beta_ss + (long long)j * p.beta_vs];
                }
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
        // ---- Pass-1 convolution of the staged raw inputs, in place, token by
        // token over the thread's channels (each thread owns its channels)
        if constexpr (CONV) {
            switch (cv.width) {
                case 1: conv_chunk<Sh, 1>(qb, kb, vb, cv_s, hist, tc, cv.silu); break;
                case 2: conv_chunk<Sh, 2>(qb, kb, vb, cv_s, hist, tc, cv.silu); break;
                case 3: conv_chunk<Sh, 3>(qb, kb, vb, cv_s, hist, tc, cv.silu); break;
                default: conv_chunk<Sh, 4>(qb, kb, vb, cv_s, hist, tc, cv.silu); break;
            }
            __syncthreads();
        }
        // ---- normalise: NL lanes per token; warp w takes tokens w, w + W, ...
        const bool rec_alpha = records && slice == 0, rec_k = rec_alpha && jr == 0;
        for (int tb = 0; tb < tc; tb += W * TPW) {
            const int tt = tb + warp + W * (lane / NL);
            const bool act = tt < tc;
            const int ts = act ? tt : 0;
            const long long rec = ring_row + (long long)(cb + ts) * rp.stride;
            norm_token<K, Sh::RPAIR, ROWS>(qb[ts], kb[ts], &sb[ts][2], lane % NL, act, p,
                                           rec_k ? rp.ring : nullptr, rp.bf16, rec);
            if (act && lane % NL == 0) {
                const float alpha = gdr_alpha(sb[ts][0], p.decay_is_log);
                sb[ts][0] = alpha;
                if (rec_alpha) ring_put1(rp.ring, rp.bf16, rec + rp.alpha_off + jr, alpha);
            }
        }
        __syncthreads();

        // ---- reductions of the chunk's first token
        const int rb = pidx<ROWS>(kl * ROWS);  // start of this lane's rows in the staged vectors
        float a[C], bq[C];
        s.partials(&kb[0][rb], &qb[0][rb], a, bq);

        // ---- the chunk's tokens
        for (int tt = 0; tt < tc; ++tt) {
            const float alpha = sb[tt][0], beta = sb[tt][1], kq = sb[tt][2];
            float u[C], o[C];
#pragma unroll
            for (int c = 0; c < C; ++c) {
                const float A = tree_lanes<LK>(a[c]);
                const float B = tree_lanes<LK>(bq[c]);
                const float bj = BPV ? b_s[bi][tt][wcol + c] : beta;
                u[c] = gdr_u(bj, alpha, A, vb[tt][wcol + c]);
                o[c] = gdr_o(alpha, B, kq, u[c]);
            }
            const int step = cb + tt;  // token index inside the row
            if (kl == 0) store_f32<C>(obase + (long long)step * p.out_ss, p.out_vs, p.out_vec, o);
            if constexpr (MODE == Mode::Verify) {
                if (records && kl == 0) {
                    const long long rec = ring_row + (long long)step * rp.stride + rp.u_off + jr * V + col0;
                    if constexpr (C % 2 == 0) {
#pragma unroll
                        for (int c = 0; c < C; c += 2) ring_put2(rp.ring, rp.bf16, rec + c, u[c], u[c + 1]);
                    } else {
#pragma unroll
                        for (int c = 0; c < C; ++c) ring_put1(rp.ring, rp.bf16, rec + c, u[c]);
                    }
                }
            }
            // One sweep: S <- k^_t u^T + alpha S, and token t+1's partials on the new S
            // (the chunk's last token sweeps against its own vectors; those partials
            // are discarded and recomputed once the next chunk is normalised).
            const int tn = tt + 1 < tc ? tt + 1 : tt;
            s.advance_partials(&kb[tt][rb], &kb[tn][rb], &qb[tn][rb], u, alpha, a, bq);
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
                            for (int c = 0; c < C; ++c) x.set(c, s.get(r, c));
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
    if (commit && p.state_out) {
        ST *sout = reinterpret_cast<ST *>(p.state_out) + soff;
#pragma unroll
        for (int i = 0; i < ROWS; ++i) {
            Pack<ST, C> x;
#pragma unroll
            for (int c = 0; c < C; ++c) x.set(c, s.get(i, c));
            x.store(sout + i * p.st_k);
        }
    }
}

// Chunk tokens of the forward pass over long or unbounded rows.
constexpr int kChainLongTC = 32;

// Batches of at most this many rows are dealt out longest row first.
constexpr int kChainOrderRows = 32;

// The launchers of each pass (one translation unit each, so they compile in
// parallel; the forward pass with V != K has its own).
cudaError_t launch_chain_fwd(const StepParams &p, int K, int V, bool bf16, long long max_len, cudaStream_t st);
cudaError_t launch_chain_fwd_kv(const StepParams &p, int K, int V, bool bf16, long long max_len, cudaStream_t st);
cudaError_t launch_chain_verify(const StepParams &p, int K, bool bf16, const RingParams &rp, long long max_len,
                                cudaStream_t st);
cudaError_t launch_chain_snap(const StepParams &p, int K, int V, bool bf16, const SnapParams &sp, long long max_len,
                              cudaStream_t st);

// Launches one instantiation with its dynamic shared memory (opted in once per
// device above 48 KiB); blocks = batch * nv * SLICES of that instantiation.
template <typename ST, int K, int V, Mode MODE, bool BPV, int TCX, bool CONV = false>
inline cudaError_t launch_chain_k(const StepParams &p, const RingParams &rp, const SnapParams &sp,
                                  long long max_len, cudaStream_t st, const ConvParams &cv = ConvParams{}) {
    using Sh = ChainShape<ST, K, V, BPV, TCX, CONV>;
    const long long blocks = (long long)p.batch * p.nv * Sh::SLICES;
    if (blocks <= 0) return cudaGetLastError();
    if (blocks >= (1ll << 31)) return cudaErrorInvalidConfiguration;
    static LaunchCache cache;
    LaunchInfo li;
    cudaError_t e = launch_info(cache, &li, [](LaunchInfo &) {
        return cudaFuncSetAttribute(k_chain<ST, K, V, MODE, BPV, TCX, CONV>,
                                    cudaFuncAttributeMaxDynamicSharedMemorySize, Sh::SMEM);
    });
    if (e != cudaSuccess) return e;
    // a few rows: deal them out longest first (chain_balanced_unit)
    const int order_p = (p.batch <= Sh::NT && p.batch <= kChainOrderRows && blocks > li.sms) ? li.sms : 0;
    k_chain<ST, K, V, MODE, BPV, TCX, CONV><<<(unsigned)blocks, Sh::NT, Sh::SMEM, st>>>(p, rp, sp, cv, max_len, order_p);
    return cudaGetLastError();
}

// The forward pass of one (state type, K, V): the chunk size follows the
// caller's row-length bound -- rows bounded at 8 or 16 tokens get chunks of
// that size (a smaller stage, more L1); longer or unbounded rows take
// kChainLongTC (fewer chunk barriers and normalisation passes per token).
template <typename ST, int K, int V>
inline cudaError_t launch_chain_fwd_t(const StepParams &p, long long max_len, cudaStream_t st) {
    const RingParams rp{};
    const SnapParams sp{};
    if (p.bpv) return launch_chain_k<ST, K, V, Mode::Fwd, true, 8>(p, rp, sp, max_len, st);
    if (max_len >= 1 && max_len <= 8) return launch_chain_k<ST, K, V, Mode::Fwd, false, 8>(p, rp, sp, max_len, st);
    if (max_len >= 1 && max_len <= 16)
        return launch_chain_k<ST, K, V, Mode::Fwd, false, 16>(p, rp, sp, max_len, st);
    return launch_chain_k<ST, K, V, Mode::Fwd, false, kChainLongTC>(p, rp, sp, max_len, st);
}

}  // namespace gdr
