// Exact fp32 CUDA-core kernels for packed-tree KDA (any of dk = dv in {32, 64, 128},
// chunk B in {16, 32, 64}).  These are the precision path: every product is fp32
// FMA, no tensor-core rounding, so fp32 workloads meet a 1e-5 relative error.  The
// tensor-core kernels (kda_seq.cu, kda_grad.cu) carry the bf16 throughput workloads.
//
// One CTA per (sequence, head) of a round.  The state S (D x D, fp32) lives in shared
// memory for the whole sequence; chunks are processed in order.  Chunk math follows
// the chunkwise form of the gated delta rule (local t = 1..L, Gamma = cumsum of g per
// channel, m = Gamma_L / 2 so that no exponential exceeds exp(|Gamma_L|/2)):
//   Kp = K e^{Gamma-m}, Km = K e^{m-Gamma}, Qp = Q e^{Gamma-m}
//   A  = strict_lower(Kp Km^T),  T = (I + diag(beta) A)^-1
//   U  = T diag(beta) (V - Kd S),          Kd = Kp e^{m}
//   O  = Qd S + incl_lower(Qp Km^T) U,     Qd = Qp e^{m}
//   S <- diag(e^{Gamma_L}) S + Kt^T U,     Kt = Km e^{Gamma_L - m}
// Replay (page "HARTS ... 精读", section 4.2): a side branch's local rows [0, rho) are
// the ancestor rows [a(p), p), gathered from the plan; they update the state but
// write no output.
#include <vector>

#include "kda_common.cuh"

namespace harts {

constexpr size_t kSimtMaxSmem = 227 * 1024;

template <int D, int BC>
struct SimtFwdLayout {
    static constexpr int kS = 0, kKp = kS + D * D, kKm = kKp + BC * D, kQp = kKm + BC * D,
                         kV = kQp + BC * D, kA = kV + BC * D, kBet = kA + BC * BC,
                         kEl = kBet + BC, kEm = kEl + D, kEkt = kEm + D, kTotal = kEkt + D;
    static constexpr size_t bytes = sizeof(float) * kTotal;
};

template <int D, int BC>
struct SimtBwdLayout {
    static constexpr int kT = BC * D, kSq = BC * BC;
    static constexpr int kS = 0, kdS = D * D, kKp = 2 * D * D, kKm = kKp + kT, kQp = kKm + kT,
                         kV = kQp + kT, kdO = kV + kT, kW1 = kdO + kT, kU = kW1 + kT,
                         kdU = kU + kT, kZ = kdU + kT, kXq = kZ + kT, kXp = kXq + kT,
                         kXm = kXp + kT, kGam = kXm + kT, kA = kGam + kT, kP = kA + kSq,
                         kdT = kP + kSq, kWm = kdT + kSq, kBet = kWm + kSq, kdBet = kBet + BC,
                         kEl = kdBet + BC, kEm = kEl + D, kEkt = kEm + D, kdGl = kEkt + D,
                         kTotal = kdGl + D;
    static constexpr size_t bytes = sizeof(float) * kTotal;
};

// Load one chunk's tiles (rows past the sequence end read as zero) and form the
// reference-scaled operands.  Gam receives the cumulative log decay.
template <int D, int BC, typename T>
__device__ void load_and_prep(const FwdParams &p, const PlanDev &pd, int32_t seq, int32_t h,
                              int32_t rho, int32_t L, int32_t c0, float *Kp, float *Km,
                              float *Qp, float *V, float *Gam, float *bet, float *el,
                              float *em, float *ekt, const T *dO_in, float *dO) {
    const int tid = threadIdx.x, nth = blockDim.x;
    const int H = p.H;
    const T *q = static_cast<const T *>(p.q), *k = static_cast<const T *>(p.k),
            *v = static_cast<const T *>(p.v), *g = static_cast<const T *>(p.g),
            *beta = static_cast<const T *>(p.beta);
    for (int i = tid; i < BC * D; i += nth) {
        const int t = i / D, c = i % D;
        const int64_t row = local_row(pd, seq, rho, L, c0 + t);
        float kk = 0.f, gg = 0.f, qq = 0.f, vv = 0.f, dd = 0.f;
        if (row >= 0) {
            const int64_t o = (row * H + h) * D + c;
            kk = ld_in(k, o); gg = ld_in(g, o); qq = ld_in(q, o) * p.scale; vv = ld_in(v, o);
            if (dO_in && c0 + t >= rho) dd = ld_in(dO_in, o);
        }
        Kp[i] = kk; Gam[i] = gg; Qp[i] = qq; V[i] = vv;
        if (dO) dO[i] = dd;
    }
    for (int t = tid; t < BC; t += nth) {
        const int64_t row = local_row(pd, seq, rho, L, c0 + t);
        bet[t] = row >= 0 ? ld_in(beta, row * H + h) : 0.f;
    }
    __syncthreads();
    for (int c = tid; c < D; c += nth) {
        float gam = 0.f;
        for (int t = 0; t < BC; ++t) { gam += Gam[t * D + c]; Gam[t * D + c] = gam; }
        const float m = 0.5f * gam;        // rows past the end hold g = 0, so gam = Gamma_L
        if (-m > kMaxExpArg) dev_error(pd, kDevErrDecayRange, seq, c0);
        for (int t = 0; t < BC; ++t) {
            const float gt = Gam[t * D + c], kk = Kp[t * D + c];
            Kp[t * D + c] = kk * expf(gt - m);
            Km[t * D + c] = kk * expf(m - gt);
            Qp[t * D + c] *= expf(gt - m);
        }
        el[c] = expf(gam);
        em[c] = expf(m);
        ekt[c] = expf(gam - m);
    }
    __syncthreads();
}

// A = strict_lower(Kp Km^T) (unscaled) in the lower triangle, then T^T in the upper
// triangle by forward substitution, one column of T per thread:
//   T_ts = -beta_t * sum_{j=s}^{t-1} A_tj T_js,   T_ss = 1.
template <int D, int BC>
__device__ void build_T(const float *Kp, const float *Km, const float *bet, float *A) {
    const int tid = threadIdx.x, nth = blockDim.x;
    for (int i = tid; i < BC * BC; i += nth) {
        const int t = i / BC, s = i % BC;
        if (s < t) {
            float acc = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) acc += Kp[t * D + c] * Km[s * D + c];
            A[i] = acc;
        }
    }
    __syncthreads();
    for (int s = tid; s < BC; s += nth) {
        for (int t = s + 1; t < BC; ++t) {
            float acc = A[t * BC + s];
            for (int j = s + 1; j < t; ++j) acc += A[t * BC + j] * A[s * BC + j];
            A[s * BC + t] = -bet[t] * acc;
        }
    }
    __syncthreads();
}

template <int D, int BC, typename T>
__global__ void __launch_bounds__(256) kda_fwd_simt(FwdParams p, PlanDev pd, int32_t round_base) {
    using Ly = SimtFwdLayout<D, BC>;
    extern __shared__ float sm[];
    float *S = sm + Ly::kS, *Kp = sm + Ly::kKp, *Km = sm + Ly::kKm, *Qp = sm + Ly::kQp,
          *V = sm + Ly::kV, *A = sm + Ly::kA, *bet = sm + Ly::kBet, *el = sm + Ly::kEl,
          *em = sm + Ly::kEm, *ekt = sm + Ly::kEkt;
    const int tid = threadIdx.x, nth = blockDim.x;
    const int H = p.H;
    const int32_t h = blockIdx.x % H;
    const int32_t seq = pd.round_order[round_base + blockIdx.x / H];
    const int32_t rho = pd.seq_rho[seq], L = rho + pd.seq_nown[seq];
    const int32_t nch = (L + BC - 1) / BC;
    const int32_t src = pd.seq_src[seq];
    const float *S0 = src >= 0 ? p.states + (static_cast<int64_t>(src) * H + h) * D * D
                    : (p.h0 ? p.h0 + (static_cast<int64_t>(-1 - src) * H + h) * D * D : nullptr);
    for (int i = tid; i < D * D; i += nth) S[i] = S0 ? S0[i] : 0.f;
    int32_t sp = pd.seq_sptr[seq];
    const int32_t sp_end = pd.seq_sptr[seq + 1];
    T *o = static_cast<T *>(p.o);
    for (int32_t ci = 0; ci < nch; ++ci) {
        const int32_t c0 = ci * BC;
        __syncthreads();
        T *rec = p.chunk_states ? static_cast<T *>(p.chunk_states) +
                     (static_cast<int64_t>(pd.seq_cbase[seq] + ci) * H + h) * (D * D + BC * BC)
                                : nullptr;
        if (rec)
            for (int i = tid; i < D * D; i += nth) st_out(rec, (i % D) * D + i / D, S[i]);
        load_and_prep<D, BC, T>(p, pd, seq, h, rho, L, c0, Kp, Km, Qp, V, Km, bet, el, em, ekt,
                                static_cast<const T *>(nullptr), nullptr);
        // load_and_prep used Km as the Gamma scratch; it is overwritten by Km itself.
        build_T<D, BC>(Kp, Km, bet, A);
        if (rec)
            for (int i = tid; i < BC * BC; i += nth) {
                const int t = i / BC, s = i % BC;
                st_out(rec + D * D, i, s < t ? A[s * BC + t] : (s == t ? 1.f : 0.f));
            }
        // Y = V - Kd S  (in place)
        for (int i = tid; i < BC * D; i += nth) {
            const int t = i / D, j = i % D;
            float acc = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) acc += Kp[t * D + c] * em[c] * S[c * D + j];
            V[i] -= acc;
        }
        __syncthreads();
        // U = T diag(beta) Y, one column per thread, rows descending (in place)
        for (int j = tid; j < D; j += nth) {
            for (int t = BC - 1; t >= 0; --t) {
                float acc = bet[t] * V[t * D + j];
                for (int s = 0; s < t; ++s) acc += A[s * BC + t] * bet[s] * V[s * D + j];
                V[t * D + j] = acc;
            }
        }
        __syncthreads();
        // P = incl_lower(Qp Km^T) into the lower triangle (T is no longer needed)
        for (int i = tid; i < BC * BC; i += nth) {
            const int t = i / BC, s = i % BC;
            if (s <= t) {
                float acc = 0.f;
#pragma unroll 8
                for (int c = 0; c < D; ++c) acc += Qp[t * D + c] * Km[s * D + c];
                A[i] = acc;
            }
        }
        __syncthreads();
        // O = Qd S + P U for own rows
        for (int i = tid; i < BC * D; i += nth) {
            const int t = i / D, j = i % D;
            if (c0 + t < rho) continue;
            const int64_t row = local_row(pd, seq, rho, L, c0 + t);
            if (row < 0) continue;
            float acc = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) acc += Qp[t * D + c] * em[c] * S[c * D + j];
            for (int s = 0; s <= t; ++s) acc += A[t * BC + s] * V[s * D + j];
            st_out(o, (row * H + h) * D + j, acc);
        }
        __syncthreads();
        // slots inside this chunk (no-replay plans): the state after the chunk's first r
        // rows, diag(e^{Gamma_{r-1}}) S + (K e^{Gamma_{r-1} - Gamma})_{<r}^T U_{<r}, as
        // e^{Gamma_{r-1} - Gamma_L} (diag(e^{Gamma_L}) S + e^{Gamma_L - m} Km_{<r}^T U_{<r}),
        // the first factor from the raw g rows r .. end of chunk
        while ((pd.flags & HARTS_PLAN_NOREPLAY) && sp < sp_end && pd.state_lpos[sp] < min(c0 + BC, L)) {
            __shared__ float s_gp[D];
            const int r = pd.state_lpos[sp] - c0;       // 1 <= r < rows of this chunk
            const int nv = min(BC, L - c0);
            for (int c = tid; c < D; c += nth) {
                float sum = 0.f;
                for (int t = r; t < nv; ++t)
                    sum += ld_in(static_cast<const T *>(p.g), (local_row(pd, seq, rho, L, c0 + t) * H + h) * D + c);
                s_gp[c] = __expf(-sum);
            }
            __syncthreads();
            float *dst = p.states + (static_cast<int64_t>(sp) * H + h) * D * D;
            for (int i = tid; i < D * D; i += nth) {
                const int c = i / D, j = i % D;
                float acc = 0.f;
                for (int t = 0; t < r; ++t) acc += Km[t * D + c] * V[t * D + j];
                dst[i] = s_gp[c] * (el[c] * S[i] + ekt[c] * acc);
            }
            __syncthreads();
            ++sp;
        }
        // S <- diag(e^{Gamma_L}) S + Kt^T U
        for (int i = tid; i < D * D; i += nth) {
            const int c = i / D, j = i % D;
            float acc = 0.f;
#pragma unroll 8
            for (int t = 0; t < BC; ++t) acc += Km[t * D + c] * V[t * D + j];
            S[i] = el[c] * S[i] + ekt[c] * acc;
        }
        __syncthreads();
        const int32_t pend = min(c0 + BC, L);     // a slot may sit at the sequence end
        if (sp < sp_end && pd.state_lpos[sp] == pend) {
            float *dst = p.states + (static_cast<int64_t>(sp) * H + h) * D * D;
            for (int i = tid; i < D * D; i += nth) dst[i] = S[i];
            ++sp;
        }
    }
    if (p.final_state) {
        float *dst = p.final_state + (static_cast<int64_t>(seq) * H + h) * D * D;
        for (int i = tid; i < D * D; i += nth) dst[i] = S[i];
    }
}

// Backward over one (sequence, head): reverse chunk loop carrying dS = dL/dS.
// Per chunk (S = chunk-start state saved by the forward, dS' = carry at chunk end):
//   dU = P^T dO + Kt dS'                Z = T^T dU            dV = beta Z
//   dT = dU (beta Y)^T (strict lower)   dM = -T^T dT T^T      dA = beta dM
//   dS <- diag(e^{Gamma_L}) dS' + Qd^T dO - (beta Kd)^T Z
// and the operand gradients are gathered per exponential factor:
//   Xq = dQd e^m + dQp,  Xp = dKd e^m + dKp,  Xm = dKm + dKt e^{Gamma_L-m}
//   dq = Xq e^{Gamma-m}, dk = Xp e^{Gamma-m} + Xm e^{m-Gamma}
//   dGamma = Xq Qp + Xp Kp - Xm Km;   dg = reverse cumsum(dGamma) + dGamma_L.
template <int D, int BC, typename T>
__global__ void __launch_bounds__(256) kda_bwd_simt(BwdParams p, PlanDev pd, int32_t round_base) {
    using Ly = SimtBwdLayout<D, BC>;
    extern __shared__ float sm[];
    float *S = sm + Ly::kS, *dS = sm + Ly::kdS, *Kp = sm + Ly::kKp, *Km = sm + Ly::kKm,
          *Qp = sm + Ly::kQp, *V = sm + Ly::kV, *dO = sm + Ly::kdO, *W1 = sm + Ly::kW1,
          *U = sm + Ly::kU, *dU = sm + Ly::kdU, *Z = sm + Ly::kZ, *Xq = sm + Ly::kXq,
          *Xp = sm + Ly::kXp, *Xm = sm + Ly::kXm, *Gam = sm + Ly::kGam, *A = sm + Ly::kA,
          *P = sm + Ly::kP, *dT = sm + Ly::kdT, *Wm = sm + Ly::kWm, *bet = sm + Ly::kBet,
          *dbet = sm + Ly::kdBet, *el = sm + Ly::kEl, *em = sm + Ly::kEm, *ekt = sm + Ly::kEkt,
          *dgl = sm + Ly::kdGl;
    const FwdParams &f = p.f;
    const int tid = threadIdx.x, nth = blockDim.x;
    const int H = f.H;
    const int32_t h = blockIdx.x % H;
    const int32_t seq = pd.round_order[round_base + blockIdx.x / H];
    const int32_t rho = pd.seq_rho[seq], L = rho + pd.seq_nown[seq];
    const int32_t nch = (L + BC - 1) / BC;
    const int32_t src = pd.seq_src[seq];
    const T *dO_in = static_cast<const T *>(p.d_o);
    T *dq = static_cast<T *>(p.dq), *dk = static_cast<T *>(p.dk), *dv = static_cast<T *>(p.dv),
      *dg = static_cast<T *>(p.dg), *db = static_cast<T *>(p.dbeta);
    for (int i = tid; i < D * D; i += nth)
        dS[i] = p.d_final ? p.d_final[(static_cast<int64_t>(seq) * H + h) * D * D + i] : 0.f;
    const int32_t sp_begin = pd.seq_sptr[seq];
    int32_t sp = pd.seq_sptr[seq + 1] - 1;
    for (int32_t ci = nch - 1; ci >= 0; --ci) {
        const int32_t c0 = ci * BC, pend = min(c0 + BC, L);
        __syncthreads();
        // consumers of the boundary state at the end of this chunk add their gradients
        if (sp >= sp_begin && pd.state_lpos[sp] == pend) {
            const int32_t cb = pd.state_cptr[sp], ce = pd.state_cptr[sp + 1];
            for (int i = tid; i < D * D; i += nth) {
                float acc = dS[i];
                for (int32_t cc = cb; cc < ce; ++cc)
                    acc += p.ds_init[(static_cast<int64_t>(pd.state_cons[cc]) * H + h) * D * D + i];
                dS[i] = acc;
            }
            --sp;
        }
        {
            const T *cs = static_cast<const T *>(f.chunk_states) +
                          (static_cast<int64_t>(pd.seq_cbase[seq] + ci) * H + h) * (D * D + BC * BC);
            for (int i = tid; i < D * D; i += nth) S[i] = ld_in(cs, (i % D) * D + i / D);
        }
        load_and_prep<D, BC, T>(f, pd, seq, h, rho, L, c0, Kp, Km, Qp, V, Gam, bet, el, em, ekt,
                                dO_in, dO);
        build_T<D, BC>(Kp, Km, bet, A);
        for (int i = tid; i < BC * BC; i += nth) {
            const int t = i / BC, s = i % BC;
            float acc = 0.f;
            if (s <= t) {
#pragma unroll 8
                for (int c = 0; c < D; ++c) acc += Qp[t * D + c] * Km[s * D + c];
            }
            P[i] = acc;
        }
        // W1 = beta (V - Kd S)
        for (int i = tid; i < BC * D; i += nth) {
            const int t = i / D, j = i % D;
            float acc = 0.f;
#pragma unroll 8
            for (int c = 0; c < D; ++c) acc += Kp[t * D + c] * em[c] * S[c * D + j];
            W1[i] = bet[t] * (V[i] - acc);
        }
        __syncthreads();
        // U = T W1;  dU = P^T dO + Kt dS'
        for (int i = tid; i < BC * D; i += nth) {
            const int t = i / D, j = i % D;
            float u = W1[i];
            for (int s = 0; s < t; ++s) u += A[s * BC + t] * W1[s * D + j];
            U[i] = u;
            float acc = 0.f;
            for (int s = t; s < BC; ++s) acc += P[s * BC + t] * dO[s * D + j];
#pragma unroll 8
            for (int c = 0; c < D; ++c) acc += Km[t * D + c] * ekt[c] * dS[c * D + j];
            dU[i] = acc;
        }
        __syncthreads();
        // Z = T^T dU;  dT = dU W1^T (strict lower)
        for (int i = tid; i < BC * D; i += nth) {
            const int t = i / D, j = i % D;
            float z = dU[i];
            for (int s = t + 1; s < BC; ++s) z += A[t * BC + s] * dU[s * D + j];
            Z[i] = z;
        }
        for (int i = tid; i < BC * BC; i += nth) {
            const int t = i / BC, s = i % BC;
            float acc = 0.f;
            if (s < t) {
#pragma unroll 8
                for (int j = 0; j < D; ++j) acc += dU[t * D + j] * W1[s * D + j];
            }
            dT[i] = acc;
        }
        __syncthreads();
        // products with S, dS', dO, U, Z
        for (int i = tid; i < BC * D; i += nth) {
            const int t = i / D, c = i % D;
            float aq = 0.f, am = 0.f, ap = 0.f;
#pragma unroll 8
            for (int j = 0; j < D; ++j) {
                aq += dO[t * D + j] * S[c * D + j];
                am += U[t * D + j] * dS[c * D + j];
                ap += Z[t * D + j] * S[c * D + j];
            }
            Xq[i] = em[c] * aq;
            Xm[i] = ekt[c] * am;
            Xp[i] = -em[c] * ap;        // dBk e^m; scaled by beta below
        }
        __syncthreads();
        // dP (incl lower) replaces P; dV = beta Z; dbeta; dGamma_L
        for (int i = tid; i < BC * BC; i += nth) {
            const int t = i / BC, s = i % BC;
            float acc = 0.f;
            if (s <= t) {
#pragma unroll 8
                for (int j = 0; j < D; ++j) acc += dO[t * D + j] * U[s * D + j];
            }
            P[i] = acc;
        }
        for (int t = tid; t < BC; t += nth) {
            float acc = 0.f;
            for (int j = 0; j < D; ++j) acc += Z[t * D + j] * V[t * D + j];
            for (int c = 0; c < D; ++c) acc += Xp[t * D + c] * Kp[t * D + c];
            dbet[t] = acc;
        }
        for (int c = tid; c < D; c += nth) {
            float acc = 0.f, ae = 0.f;
            for (int t = 0; t < BC; ++t) acc += Xm[t * D + c] * Km[t * D + c];
            for (int j = 0; j < D; ++j) ae += S[c * D + j] * dS[c * D + j];
            dgl[c] = acc + el[c] * ae;
        }
        __syncthreads();
        // carry: dS <- el dS' + Qd^T dO - (beta Kd)^T Z   (in place, per element)
        for (int i = tid; i < D * D; i += nth) {
            const int c = i / D, j = i % D;
            float a1 = 0.f, a2 = 0.f;
            for (int t = 0; t < BC; ++t) {
                a1 += Qp[t * D + c] * dO[t * D + j];
                a2 += bet[t] * Kp[t * D + c] * Z[t * D + j];
            }
            dS[i] = el[c] * dS[i] + em[c] * (a1 - a2);
        }
        for (int i = tid; i < BC * D; i += nth) Xp[i] *= bet[i / D];
        // Wm = dT T^T
        for (int i = tid; i < BC * BC; i += nth) {
            const int t = i / BC, s = i % BC;
            const int jmax = min(s, t - 1);
            float acc = 0.f;
            for (int j = 0; j <= jmax; ++j) acc += dT[t * BC + j] * (j == s ? 1.f : A[j * BC + s]);
            Wm[i] = acc;
        }
        __syncthreads();
        // dM = -T^T Wm (strict lower) -> dA = beta dM into dT; dbeta += sum_b dM A
        for (int a = tid; a < BC; a += nth) {
            float dba = 0.f;
            for (int b = 0; b < a; ++b) {
                float acc = Wm[a * BC + b];
                for (int t = a + 1; t < BC; ++t) acc += A[a * BC + t] * Wm[t * BC + b];
                const float dm = -acc;
                dba += dm * A[a * BC + b];
                dT[a * BC + b] = bet[a] * dm;
            }
            for (int b = a; b < BC; ++b) dT[a * BC + b] = 0.f;
            dbet[a] += dba;
        }
        __syncthreads();
        // Xp += dA Km;  Xm += dA^T Kp + dP^T Qp;  Xq += dP Km
        for (int i = tid; i < BC * D; i += nth) {
            const int t = i / D, c = i % D;
            float ap = 0.f, aq = 0.f, am = 0.f;
            for (int s = 0; s < BC; ++s) {
                const float km = Km[s * D + c];
                ap += dT[t * BC + s] * km;
                aq += P[t * BC + s] * km;
                am += dT[s * BC + t] * Kp[s * D + c] + P[s * BC + t] * Qp[s * D + c];
            }
            Xp[i] += ap;
            Xq[i] += aq;
            Xm[i] += am;
        }
        __syncthreads();
        // outputs
        for (int c = tid; c < D; c += nth) {
            // the reference m = Gamma_L / 2, recovered from the last row of Gam
            const float mref = 0.5f * Gam[(BC - 1) * D + c];
            float run = dgl[c];
            for (int t = BC - 1; t >= 0; --t) {
                const int i = t * D + c;
                const float dgam = Xq[i] * Qp[i] + Xp[i] * Kp[i] - Xm[i] * Km[i];
                run += dgam;
                const float ep = expf(Gam[i] - mref), en = expf(mref - Gam[i]);
                const float dkk = Xp[i] * ep + Xm[i] * en;
                const float dqq = Xq[i] * ep * f.scale;
                const int32_t r = c0 + t;
                if (r >= L) continue;
                const int64_t row = local_row(pd, seq, rho, L, r);
                if (r >= rho) {
                    const int64_t o = (row * H + h) * D + c;
                    st_out(dq, o, dqq); st_out(dk, o, dkk); st_out(dg, o, run);
                } else {
                    float *rg = p.rep_grad + (static_cast<int64_t>(pd.seq_rptr[seq] + r) * H + h) * rep_width(D);
                    rg[c] = dkk; rg[2 * D + c] = run;
                }
            }
        }
        for (int i = tid; i < BC * D; i += nth) {
            const int t = i / D, j = i % D;
            const int32_t r = c0 + t;
            if (r >= L) continue;
            const float x = bet[t] * Z[i];
            if (r >= rho) {
                const int64_t row = local_row(pd, seq, rho, L, r);
                st_out(dv, (row * H + h) * D + j, x);
            } else {
                p.rep_grad[(static_cast<int64_t>(pd.seq_rptr[seq] + r) * H + h) * rep_width(D) + D + j] = x;
            }
        }
        for (int t = tid; t < BC; t += nth) {
            const int32_t r = c0 + t;
            if (r >= L) continue;
            if (r >= rho) {
                const int64_t row = local_row(pd, seq, rho, L, r);
                st_out(db, row * H + h, dbet[t]);
            } else {
                p.rep_grad[(static_cast<int64_t>(pd.seq_rptr[seq] + r) * H + h) * rep_width(D) + 3 * D] = dbet[t];
            }
        }
    }
    __syncthreads();
    if (src >= 0 || p.dh0) {
        float *dst = p.ds_init + (static_cast<int64_t>(seq) * H + h) * D * D;
        for (int i = tid; i < D * D; i += nth) dst[i] = dS[i];
    }
}

// Deterministic fold of replay-row gradients into their compact rows: per distinct
// replayed row, occurrences are summed in ascending occurrence order, then added.
template <typename T>
__global__ void fold_replay_grads(BwdParams p, PlanDev pd, int D) {
    // one block per ancestor row that replayed rows copy, all heads; each thread sums 4
    // consecutive floats of a head's replay-gradient rows over the row's occurrences (in
    // ascending occurrence order) and adds them to the row's dk, dv, dg, dbeta
    const int32_t f = blockIdx.x, H = p.f.H;
    const int32_t row = pd.fold_rows[f];
    const int W = rep_width(D), W4 = W / 4;
    const int32_t j0 = pd.fold_ptr[f], j1 = pd.fold_ptr[f + 1];
    T *dk = static_cast<T *>(p.dk), *dv = static_cast<T *>(p.dv), *dg = static_cast<T *>(p.dg),
      *db = static_cast<T *>(p.dbeta);
    for (int u = threadIdx.x; u < H * W4; u += blockDim.x) {
        const int h = u / W4, e4 = u - h * W4;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        for (int32_t j = j0; j < j1; ++j) {
            const float4 x = reinterpret_cast<const float4 *>(
                p.rep_grad + (static_cast<int64_t>(pd.fold_occ[j]) * H + h) * W)[e4];
            acc.x += x.x; acc.y += x.y; acc.z += x.z; acc.w += x.w;
        }
        const int64_t rh = static_cast<int64_t>(row) * H + h;
        const float a[4] = {acc.x, acc.y, acc.z, acc.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int e = 4 * e4 + i;
            if (e < D) st_out(dk, rh * D + e, ld_in(dk, rh * D + e) + a[i]);
            else if (e < 2 * D) st_out(dv, rh * D + e - D, ld_in(dv, rh * D + e - D) + a[i]);
            else if (e < 3 * D) st_out(dg, rh * D + e - 2 * D, ld_in(dg, rh * D + e - 2 * D) + a[i]);
            else if (e == 3 * D) st_out(db, rh, ld_in(db, rh) + a[i]);
        }
    }
}

// dh0[r] = sum of the initial-state gradients of every sequence that starts from root r.
__global__ void reduce_dh0(BwdParams p, PlanDev pd, int D) {
    const int32_t r = blockIdx.x, h = blockIdx.y, H = p.f.H;
    for (int i = threadIdx.x; i < D * D; i += blockDim.x) {
        float acc = 0.f;
        for (int32_t j = pd.root_cptr[r]; j < pd.root_cptr[r + 1]; ++j)
            acc += p.ds_init[(static_cast<int64_t>(pd.root_cons[j]) * H + h) * D * D + i];
        p.dh0[(static_cast<int64_t>(r) * H + h) * D * D + i] = acc;
    }
}

// ---- launchers ---------------------------------------------------------------------

template <int D, int BC, typename T>
static cudaError_t fwd_t(const FwdParams &p, const PlanDev &pd, int32_t base, int32_t n_items,
                         cudaStream_t st) {
    using Ly = SimtFwdLayout<D, BC>;
    auto kern = kda_fwd_simt<D, BC, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Ly::bytes));
    if (e != cudaSuccess) return e;
    kern<<<n_items, 256, Ly::bytes, st>>>(p, pd, base);
    return cudaGetLastError();
}

template <int D, int BC, typename T>
static cudaError_t bwd_t(const BwdParams &p, const PlanDev &pd, int32_t base, int32_t n_items,
                         cudaStream_t st) {
    using Ly = SimtBwdLayout<D, BC>;
    if (Ly::bytes > kSimtMaxSmem) return cudaErrorInvalidConfiguration;
    auto kern = kda_bwd_simt<D, BC, T>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         static_cast<int>(Ly::bytes));
    if (e != cudaSuccess) return e;
    kern<<<n_items, 256, Ly::bytes, st>>>(p, pd, base);
    return cudaGetLastError();
}

template <typename T>
static cudaError_t fwd_dispatch(int D, int BC, const FwdParams &p, const PlanDev &pd,
                                int32_t base, int32_t n, cudaStream_t st) {
#define HARTS_CASE(d, b) if (D == d && BC == b) return fwd_t<d, b, T>(p, pd, base, n, st);
    HARTS_CASE(32, 16) HARTS_CASE(32, 32) HARTS_CASE(32, 64)
    HARTS_CASE(64, 16) HARTS_CASE(64, 32) HARTS_CASE(64, 64)
    HARTS_CASE(128, 16) HARTS_CASE(128, 32) HARTS_CASE(128, 64)
#undef HARTS_CASE
    return cudaErrorInvalidValue;
}

template <typename T>
static cudaError_t bwd_dispatch(int D, int BC, const BwdParams &p, const PlanDev &pd,
                                int32_t base, int32_t n, cudaStream_t st) {
#define HARTS_CASE(d, b) if (D == d && BC == b) return bwd_t<d, b, T>(p, pd, base, n, st);
    HARTS_CASE(32, 16) HARTS_CASE(32, 32) HARTS_CASE(32, 64)
    HARTS_CASE(64, 16) HARTS_CASE(64, 32)
#undef HARTS_CASE
    return cudaErrorInvalidValue;
}

bool simt_supported(bool backward, int D, int BC) {
    if (!(D == 32 || D == 64 || D == 128) || !(BC == 16 || BC == 32 || BC == 64)) return false;
    if (!backward) return true;
    return D == 32 || (D == 64 && BC <= 32);
}

cudaError_t simt_fwd_round(int dtype, int BC, const FwdParams &p, const PlanDev &pd,
                           int32_t base, int32_t n_items, cudaStream_t st) {
    return dtype == HARTS_FP32 ? fwd_dispatch<float>(p.D, BC, p, pd, base, n_items, st)
                               : fwd_dispatch<__nv_bfloat16>(p.D, BC, p, pd, base, n_items, st);
}

cudaError_t simt_bwd_round(int dtype, int BC, const BwdParams &p, const PlanDev &pd,
                           int32_t base, int32_t n_items, cudaStream_t st) {
    return dtype == HARTS_FP32 ? bwd_dispatch<float>(p.f.D, BC, p, pd, base, n_items, st)
                               : bwd_dispatch<__nv_bfloat16>(p.f.D, BC, p, pd, base, n_items, st);
}

cudaError_t bwd_finish(int dtype, const BwdParams &p, const PlanDev &pd, cudaStream_t st) {
    const int D = p.f.D, H = p.f.H;
    if (pd.n_fold > 0) {
        if (dtype == HARTS_FP32) fold_replay_grads<float><<<pd.n_fold, 256, 0, st>>>(p, pd, D);
        else fold_replay_grads<__nv_bfloat16><<<pd.n_fold, 256, 0, st>>>(p, pd, D);
        cudaError_t e = cudaGetLastError();
        if (e != cudaSuccess) return e;
    }
    if (p.dh0 && pd.n_roots > 0) {
        reduce_dh0<<<dim3(pd.n_roots, H), 256, 0, st>>>(p, pd, D);
        return cudaGetLastError();
    }
    return cudaSuccess;
}

}  // namespace harts
