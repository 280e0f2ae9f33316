/*
 * wkv7_oracle.c -- plain, slow fp64 reference of the WKV7 state recurrence.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, includes or
 * calls this file; only the tests, the smoke check and the CPU-baseline leg of
 * the benchmark load it.  It shares no code with the CUDA path.
 *
 * What it computes (per batch row b and head h; state S is D x D, row i is the
 * value index, column j the key index):
 *
 *   sa_i   = sum_j S_ij a_j                          (uses the state before the update)
 *   S_ij  <- S_ij w_j + v_i k_j + sa_i b_j
 *   y_i    = sum_j S_ij r_j                          (uses the updated state)
 *
 * Source: "RWKV-7 Pretraining on Apple Silicon (MLX)", section "Metal kernel
 * architecture", Forward listing (h = w*h + v*k + sa*b; y = dot(h, r); a
 * checkpoint of h after every chunk of 32 tokens).  The listing leaves `sa`
 * undefined; it is read as the state times a, taken before the update.
 *
 * Backward: reverse-mode differentiation of the forward, token by token in
 * reverse ("Backward" listing of the same section: VJP for dr, dw, dk, dv, da,
 * db, walking chunks in reverse from the exact checkpoints).  With G the
 * gradient of the loss w.r.t. the state after token t (incoming from later
 * tokens), per token in reverse:
 *
 *   G_ij  += dy_i r_j
 *   dr_j   = sum_i dy_i S'_ij        (S' = state after the update)
 *   dw_j   = sum_i G_ij S_ij         (S  = state before the update)
 *   dk_j   = sum_i G_ij v_i
 *   dv_i   = sum_j G_ij k_j
 *   db_j   = sum_i G_ij sa_i
 *   dsa_i  = sum_j G_ij b_j
 *   da_j   = sum_i dsa_i S_ij
 *   G_ij  <- G_ij w_j + dsa_i a_j    (gradient w.r.t. the state before the update)
 *
 * Three ways to obtain S and sa in the reverse walk are kept, for the checks:
 *   full : every state of the forward is stored (small problems only);
 *   ckpt : each chunk is recomputed forward from its start checkpoint and its
 *          states are kept (exact, any size);
 *   recon: the page's reconstruction S = (S' - v k^T - sa b^T) / w (column j
 *          divided by w_j), starting from the chunk-end checkpoint, with sa
 *          recomputed forward from the chunk-start checkpoint.
 *
 * Checkpoints: C = ceil(T / chunk) entries; entry c is the state after token
 * min(T, (c+1)*chunk) - 1, so the last entry equals hT.
 *
 * Layouts (row-major): per-token tensors (B, T, H, D); states (B, H, D, D);
 * checkpoints (B, H, C, D, D).  All arithmetic is fp64, one thread, no
 * blocking, fusion or reordering beyond the definitions above.
 */
#include <stdlib.h>
#include <string.h>

static size_t tix(int b, int t, int h, int T, int H, int D)
{
    return (((size_t)b * T + t) * H + h) * (size_t)D;
}

static size_t six(int b, int h, int H, int D)
{
    return ((size_t)b * H + h) * (size_t)D * D;
}

/* one token of the forward on one head: S is updated in place, sa receives S a */
static void step_forward(int D, double *S, double *sa,
                         const double *w, const double *k, const double *v,
                         const double *a, const double *bb)
{
    for (int i = 0; i < D; i++) {
        double s = 0.0;
        for (int j = 0; j < D; j++) s += S[i * D + j] * a[j];
        sa[i] = s;
    }
    for (int i = 0; i < D; i++)
        for (int j = 0; j < D; j++)
            S[i * D + j] = S[i * D + j] * w[j] + v[i] * k[j] + sa[i] * bb[j];
}

int wkv7_oracle_num_chunks(int T, int chunk) { return (T + chunk - 1) / chunk; }

/* forward: y (B,T,H,D); h_ckpt (B,H,C,D,D) or NULL; hT (B,H,D,D) or NULL; h0 NULL = zeros;
 * sa_out (B,T,H,D) or NULL receives sa_t = S_{t-1} a_t of every token and row */
int wkv7_oracle_forward(int B, int T, int H, int D, int chunk,
                        const double *r, const double *w, const double *k,
                        const double *v, const double *a, const double *bb,
                        const double *h0, double *y, double *h_ckpt, double *hT, double *sa_out)
{
    if (B < 0 || T < 0 || H < 0 || D <= 0 || chunk <= 0) return 1;
    const int C = wkv7_oracle_num_chunks(T, chunk);
    double *S = (double *)malloc(sizeof(double) * D * D);
    double *sa = (double *)malloc(sizeof(double) * D);
    if (!S || !sa) { free(S); free(sa); return 2; }
    for (int b = 0; b < B; b++)
        for (int h = 0; h < H; h++) {
            if (h0) memcpy(S, h0 + six(b, h, H, D), sizeof(double) * D * D);
            else memset(S, 0, sizeof(double) * D * D);
            for (int t = 0; t < T; t++) {
                size_t o = tix(b, t, h, T, H, D);
                step_forward(D, S, sa, w + o, k + o, v + o, a + o, bb + o);
                if (sa_out) memcpy(sa_out + o, sa, sizeof(double) * D);
                for (int i = 0; i < D; i++) {
                    double s = 0.0;
                    for (int j = 0; j < D; j++) s += S[i * D + j] * r[o + j];
                    y[o + i] = s;
                }
                if (h_ckpt && ((t + 1) % chunk == 0 || t == T - 1)) {
                    size_t co = (((size_t)b * H + h) * C + t / chunk) * (size_t)D * D;
                    memcpy(h_ckpt + co, S, sizeof(double) * D * D);
                }
            }
            if (hT) memcpy(hT + six(b, h, H, D), S, sizeof(double) * D * D);
        }
    free(S);
    free(sa);
    return 0;
}

/* single-token decode: state (B,H,D,D) updated in place; inputs (B,H,D); y (B,H,D) */
int wkv7_oracle_decode(int B, int H, int D, double *state,
                       const double *r, const double *w, const double *k,
                       const double *v, const double *a, const double *bb, double *y)
{
    return wkv7_oracle_forward(B, 1, H, D, 1, r, w, k, v, a, bb, state, y, NULL, state, NULL);
}

/* reverse walk over tokens t1-1 .. t0 of one head.  states[t - t0] is the state before
 * token t (t0 <= t <= t1, so states has t1-t0+1 entries, the last being the state after
 * token t1-1) -- used when `states` is non-NULL.  Otherwise (recon) Scur holds the state
 * after token t1-1 on entry and the page's reconstruction is applied; sas[t - t0] = sa_t. */
static void reverse_walk(int b, int h, int T, int H, int D, int t0, int t1,
                         const double *r, const double *w, const double *k,
                         const double *v, const double *a, const double *bb,
                         const double *dy, const double *states, double *Scur,
                         const double *sas, double *G, double *Sprev, double *dsa,
                         double *dr, double *dw, double *dk, double *dv, double *da, double *db)
{
    for (int t = t1 - 1; t >= t0; t--) {
        size_t o = tix(b, t, h, T, H, D);
        const double *sa = sas + (size_t)(t - t0) * D;
        const double *Snew;
        const double *S;
        if (states) {
            Snew = states + (size_t)(t - t0 + 1) * D * D;
            S = states + (size_t)(t - t0) * D * D;
        } else {
            Snew = Scur;
            for (int i = 0; i < D; i++)
                for (int j = 0; j < D; j++)
                    Sprev[i * D + j] = (Scur[i * D + j] - v[o + i] * k[o + j] - sa[i] * bb[o + j]) / w[o + j];
            S = Sprev;
        }
        for (int i = 0; i < D; i++)
            for (int j = 0; j < D; j++) G[i * D + j] += dy[o + i] * r[o + j];
        for (int j = 0; j < D; j++) {
            double s_r = 0.0, s_w = 0.0, s_k = 0.0, s_b = 0.0;
            for (int i = 0; i < D; i++) {
                s_r += dy[o + i] * Snew[i * D + j];
                s_w += G[i * D + j] * S[i * D + j];
                s_k += G[i * D + j] * v[o + i];
                s_b += G[i * D + j] * sa[i];
            }
            dr[o + j] = s_r;
            dw[o + j] = s_w;
            dk[o + j] = s_k;
            db[o + j] = s_b;
        }
        for (int i = 0; i < D; i++) {
            double s_v = 0.0, s_sa = 0.0;
            for (int j = 0; j < D; j++) {
                s_v += G[i * D + j] * k[o + j];
                s_sa += G[i * D + j] * bb[o + j];
            }
            dv[o + i] = s_v;
            dsa[i] = s_sa;
        }
        for (int j = 0; j < D; j++) {
            double s = 0.0;
            for (int i = 0; i < D; i++) s += dsa[i] * S[i * D + j];
            da[o + j] = s;
        }
        for (int i = 0; i < D; i++)
            for (int j = 0; j < D; j++) G[i * D + j] = G[i * D + j] * w[o + j] + dsa[i] * a[o + j];
        if (!states) memcpy(Scur, Sprev, sizeof(double) * D * D);
    }
}

/* mode 0 = full (stores all states), 1 = ckpt (exact chunk recompute),
 * 2 = recon (page reconstruction from the chunk-end checkpoint).
 * h_ckpt is required for modes 1 and 2 (as written by the forward); h0, dhT, dh0 may be NULL. */
int wkv7_oracle_backward(int mode, int B, int T, int H, int D, int chunk,
                         const double *r, const double *w, const double *k,
                         const double *v, const double *a, const double *bb,
                         const double *h0, const double *h_ckpt,
                         const double *dy, const double *dhT,
                         double *dr, double *dw, double *dk, double *dv, double *da, double *db,
                         double *dh0)
{
    if (B < 0 || T < 0 || H < 0 || D <= 0 || chunk <= 0 || mode < 0 || mode > 2) return 1;
    if (mode != 0 && !h_ckpt && T > 0) return 1;
    const int C = wkv7_oracle_num_chunks(T, chunk);
    const int span = mode == 0 ? T : chunk;     /* tokens whose states are kept at once */
    const size_t DD = (size_t)D * D;
    double *states = (double *)malloc(sizeof(double) * DD * (size_t)(span + 1));
    double *sas = (double *)malloc(sizeof(double) * D * (size_t)(span > 0 ? span : 1));
    double *G = (double *)malloc(sizeof(double) * DD);
    double *Scur = (double *)malloc(sizeof(double) * DD);
    double *Sprev = (double *)malloc(sizeof(double) * DD);
    double *dsa = (double *)malloc(sizeof(double) * D);
    if (!states || !sas || !G || !Scur || !Sprev || !dsa) {
        free(states); free(sas); free(G); free(Scur); free(Sprev); free(dsa);
        return 2;
    }
    for (int b = 0; b < B; b++)
        for (int h = 0; h < H; h++) {
            if (dhT) memcpy(G, dhT + six(b, h, H, D), sizeof(double) * DD);
            else memset(G, 0, sizeof(double) * DD);
            const int first_c = mode == 0 ? 0 : C - 1;
            for (int c = first_c; c >= 0; c--) {
                const int t0 = mode == 0 ? 0 : c * chunk;
                const int t1 = mode == 0 ? T : (t0 + chunk < T ? t0 + chunk : T);
                /* state before token t0 */
                double *S = states;
                if (t0 == 0) {
                    if (h0) memcpy(S, h0 + six(b, h, H, D), sizeof(double) * DD);
                    else memset(S, 0, sizeof(double) * DD);
                } else {
                    size_t co = (((size_t)b * H + h) * C + (c - 1)) * DD;
                    memcpy(S, h_ckpt + co, sizeof(double) * DD);
                }
                /* forward over the span, keeping every state and every sa */
                for (int t = t0; t < t1; t++) {
                    size_t o = tix(b, t, h, T, H, D);
                    double *Sn = states + (size_t)(t - t0 + 1) * DD;
                    memcpy(Sn, states + (size_t)(t - t0) * DD, sizeof(double) * DD);
                    step_forward(D, Sn, sas + (size_t)(t - t0) * D, w + o, k + o, v + o, a + o, bb + o);
                }
                if (mode == 2) {
                    size_t co = (((size_t)b * H + h) * C + c) * DD;
                    memcpy(Scur, h_ckpt + co, sizeof(double) * DD);
                    reverse_walk(b, h, T, H, D, t0, t1, r, w, k, v, a, bb, dy, NULL, Scur, sas,
                                 G, Sprev, dsa, dr, dw, dk, dv, da, db);
                } else {
                    reverse_walk(b, h, T, H, D, t0, t1, r, w, k, v, a, bb, dy, states, NULL, sas,
                                 G, Sprev, dsa, dr, dw, dk, dv, da, db);
                }
            }
            if (dh0) memcpy(dh0 + six(b, h, H, D), G, sizeof(double) * DD);
        }
    free(states); free(sas); free(G); free(Scur); free(Sprev); free(dsa);
    return 0;
}
