// Plain fp64 C++ oracle of the fused top-K forward-KL distillation loss.
//
// TEST INFRASTRUCTURE ONLY.  Only the tests, the package smoke check and the
// benchmark's CPU legs load this library; the CUDA path shares no code with it.
//
// It is the definition written out with loops, one full logit row of length V
// at a time, with no blocking, fusion or reordering beyond that:
//
//   teacher   p_ik = exp(t_ik/T - max_k t/T) / sum_k exp(...)   over the K cached
//             entries only (renormalised); -inf logits carry p = 0 and 0 log 0 = 0.
//             The cache holds the teacher's top-100 per position: "Effektivnaya
//             distillyatsiya znaniy" (malakhovai.ru), paragraph 2, and
//             "Wissensdestillation mit deutlich weniger GPU-Speicher"
//             (dailytechsnack.ch), section "Teacher-Ausgaben einmalig
//             zwischenspeichern".  Both sides are divided by T before the softmax:
//             "Distillyatsiya i szhatie modeley" (ml-book.com), section "Kak eto
//             rabotaet: myagkie metki i temperatura".
//   student   z_iv = sum_j h_ij W_vj for every v of the full vocabulary,
//             a = z/T, lse_i = m + log sum_v exp(a_iv - m) with m = max_v a_iv.
//   loss      KL_i = sum_k p_ik (log p_ik - (a_{i,idx_ik} - lse_i)),
//             loss = T^2 sum_{valid i} KL_i / N_valid   (same ml-book.com section:
//             the T^2 factor restores the gradient scale), 0 if N_valid = 0.
//   gradient  dz_iv = valid_i g T (exp(a_iv - lse_i) - s_iv) / N_valid with
//             s_iv = sum_{k: idx_ik = v} p_ik; dh_i = sum_v dz_iv W_v and
//             dW_v = sum_i dz_iv h_i (rows summed in increasing order).
//
// A row is valid when its mask byte is non-zero (or mask is NULL) and at least
// one of its teacher logits is finite.
//
// Threads only split independent outputs (rows for z / lse / KL / dh, vocabulary
// rows for dW); every output element is summed by one thread in a fixed order,
// so results do not depend on the thread count or on row_block.
#include <algorithm>
#include <cmath>
#include <numeric>
#include <cstdint>
#include <limits>
#include <thread>
#include <vector>

namespace {

constexpr double kNegInf = -std::numeric_limits<double>::infinity();

template <class F>
void parallel_for(int64_t n, int threads, F f) {
    if (threads < 1) threads = 1;
    if (threads > n) threads = static_cast<int>(std::max<int64_t>(n, 1));
    if (threads == 1) {
        f(0, n);
        return;
    }
    std::vector<std::thread> pool;
    for (int t = 0; t < threads; ++t) {
        const int64_t b = n * t / threads, e = n * (t + 1) / threads;
        pool.emplace_back([=] { f(b, e); });
    }
    for (auto& th : pool) th.join();
}

// p over the K cached entries of one row; returns whether any logit is finite.
bool teacher_row(const double* t, int64_t K, double T, double* p) {
    double m = kNegInf;
    for (int64_t k = 0; k < K; ++k)
        if (std::isfinite(t[k])) m = std::max(m, t[k] / T);
    if (m == kNegInf) {
        for (int64_t k = 0; k < K; ++k) p[k] = 0.0;
        return false;
    }
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        p[k] = std::isfinite(t[k]) ? std::exp(t[k] / T - m) : 0.0;
        s += p[k];
    }
    for (int64_t k = 0; k < K; ++k) p[k] /= s;
    return true;
}

bool row_valid(const uint8_t* mask, int64_t i, bool has_mass) {
    return (mask == nullptr || mask[i] != 0) && has_mass;
}

// One full logit row: z[v] = sum_j h_i[j] W[v][j].
void logit_row(const double* hi, const double* W, int64_t d, int64_t V, double* z) {
    for (int64_t v = 0; v < V; ++v) {
        const double* wv = W + v * d;
        double acc = 0.0;
        for (int64_t j = 0; j < d; ++j) acc += hi[j] * wv[j];
        z[v] = acc;
    }
}

// lse of a = z/T over the whole row.
double lse_row(const double* z, int64_t V, double T) {
    double m = kNegInf;
    for (int64_t v = 0; v < V; ++v) m = std::max(m, z[v] / T);
    double s = 0.0;
    for (int64_t v = 0; v < V; ++v) s += std::exp(z[v] / T - m);
    return m + std::log(s);
}

// KL_i from the materialised row.
double kl_row(const double* z, const int32_t* idx, const double* p, int64_t K, double T, double lse) {
    double kl = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        if (p[k] > 0.0) {
            const double logq = z[idx[k]] / T - lse;
            kl += p[k] * (std::log(p[k]) - logq);
        }
    }
    return kl;
}

// dz row = coef (q - s).
void dz_row(const double* z, const int32_t* idx, const double* p, int64_t V, int64_t K, double T,
            double lse, double coef, double* dz) {
    for (int64_t v = 0; v < V; ++v) dz[v] = std::exp(z[v] / T - lse);
    for (int64_t k = 0; k < K; ++k) dz[idx[k]] -= p[k];
    for (int64_t v = 0; v < V; ++v) dz[v] *= coef;
}

// The forward of one row: its full logit row z, lse (at T) and KL.
void forward_row(const double* hi, const double* W, const int32_t* idx_i, const double* p, int64_t d, int64_t V,
                 int64_t K, double T, double* z, double* lse, double* kl) {
    logit_row(hi, W, d, V, z);
    *lse = lse_row(z, V, T);
    *kl = kl_row(z, idx_i, p, K, T, *lse);
}

// dh_i += sum_v dz_iv W_v.
void add_dh_row(const double* dzr, const double* W, int64_t V, int64_t d, double* dhi) {
    for (int64_t v = 0; v < V; ++v)
        for (int64_t j = 0; j < d; ++j) dhi[j] += dzr[v] * W[v * d + j];
}

int64_t count_valid(const double* t, const uint8_t* mask, int64_t N, int64_t K, double T) {
    std::vector<double> p(static_cast<size_t>(K));
    int64_t n = 0;
    for (int64_t i = 0; i < N; ++i) n += row_valid(mask, i, teacher_row(t + i * K, K, T, p.data())) ? 1 : 0;
    return n;
}

}  // namespace

extern "C" {

// p [N][K] and has_mass [N] (0/1).
void fklo_teacher(const double* t, int64_t N, int64_t K, double T, double* p, uint8_t* has_mass) {
    for (int64_t i = 0; i < N; ++i) has_mass[i] = teacher_row(t + i * K, K, T, p + i * K) ? 1 : 0;
}

// lse [N], kl [N], valid [N]; *loss and *n_valid.
void fklo_forward(const double* h, const double* W, const int32_t* idx, const double* t, const uint8_t* mask,
                  int64_t N, int64_t d, int64_t V, int64_t K, double T, int threads, double* lse, double* kl,
                  uint8_t* valid, double* loss, int64_t* n_valid) {
    parallel_for(N, threads, [&](int64_t b, int64_t e) {
        std::vector<double> z(static_cast<size_t>(V)), p(static_cast<size_t>(K));
        for (int64_t i = b; i < e; ++i) {
            const bool has = teacher_row(t + i * K, K, T, p.data());
            valid[i] = row_valid(mask, i, has) ? 1 : 0;
            forward_row(h + i * d, W, idx + i * K, p.data(), d, V, K, T, z.data(), lse + i, kl + i);
        }
    });
    int64_t nv = 0;
    double sum = 0.0;
    for (int64_t i = 0; i < N; ++i) {
        if (valid[i]) {
            ++nv;
            sum += kl[i];
        }
    }
    *n_valid = nv;
    *loss = nv > 0 ? T * T * sum / static_cast<double>(nv) : 0.0;
}

// dh [N][d] and dW [V][d], both overwritten.  Rows are taken in blocks of
// row_block: the block's dz rows are materialised, then dh of those rows and
// their contribution to every dW row (added in increasing row order).
void fklo_backward(const double* h, const double* W, const int32_t* idx, const double* t, const uint8_t* mask,
                   int64_t N, int64_t d, int64_t V, int64_t K, double T, double grad_loss, int64_t row_block,
                   int threads, double* dh, double* dW) {
    std::fill(dh, dh + N * d, 0.0);
    std::fill(dW, dW + V * d, 0.0);
    const int64_t nv = count_valid(t, mask, N, K, T);
    if (nv == 0) return;
    if (row_block < 1) row_block = 1;
    std::vector<double> dz(static_cast<size_t>(row_block * V));
    for (int64_t r0 = 0; r0 < N; r0 += row_block) {
        const int64_t r1 = std::min(N, r0 + row_block);
        parallel_for(r1 - r0, threads, [&](int64_t b, int64_t e) {
            std::vector<double> z(static_cast<size_t>(V)), p(static_cast<size_t>(K));
            for (int64_t r = b; r < e; ++r) {
                const int64_t i = r0 + r;
                const bool has = teacher_row(t + i * K, K, T, p.data());
                const double coef = row_valid(mask, i, has) ? grad_loss * T / static_cast<double>(nv) : 0.0;
                double* dzr = dz.data() + r * V;
                logit_row(h + i * d, W, d, V, z.data());
                dz_row(z.data(), idx + i * K, p.data(), V, K, T, lse_row(z.data(), V, T), coef, dzr);
                add_dh_row(dzr, W, V, d, dh + i * d);
            }
        });
        parallel_for(V, threads, [&](int64_t b, int64_t e) {
            for (int64_t v = b; v < e; ++v) {
                double* dwv = dW + v * d;
                for (int64_t i = r0; i < r1; ++i) {
                    const double c = dz[(i - r0) * V + v];
                    for (int64_t j = 0; j < d; ++j) dwv[j] += c * h[i * d + j];
                }
            }
        });
    }
}

// lse, KL and dh of the rows listed in `rows` (n of them); N_valid is counted
// over all N rows.  Outputs are [n], [n], [n][d].
void fklo_rows(const double* h, const double* W, const int32_t* idx, const double* t, const uint8_t* mask,
               int64_t N, int64_t d, int64_t V, int64_t K, double T, double grad_loss, const int64_t* rows,
               int64_t n, int threads, double* lse, double* kl, double* dh, int64_t* n_valid) {
    const int64_t nv = count_valid(t, mask, N, K, T);
    *n_valid = nv;
    parallel_for(n, threads, [&](int64_t b, int64_t e) {
        std::vector<double> z(static_cast<size_t>(V)), p(static_cast<size_t>(K)), dz(static_cast<size_t>(V));
        for (int64_t r = b; r < e; ++r) {
            const int64_t i = rows[r];
            const bool has = teacher_row(t + i * K, K, T, p.data());
            forward_row(h + i * d, W, idx + i * K, p.data(), d, V, K, T, z.data(), lse + r, kl + r);
            double* dhr = dh + r * d;
            std::fill(dhr, dhr + d, 0.0);
            if (nv == 0) continue;
            const double coef = row_valid(mask, i, has) ? grad_loss * T / static_cast<double>(nv) : 0.0;
            dz_row(z.data(), idx + i * K, p.data(), V, K, T, lse[r], coef, dz.data());
            add_dh_row(dz.data(), W, V, d, dhr);
        }
    });
}

// dW restricted to the vocabulary rows `vrows` (nv_rows of them), given the
// per-token lse [N]: out[r] = sum_i dz_{i, vrows[r]} h_i.
void fklo_dW_rows(const double* h, const double* W, const int32_t* idx, const double* t, const uint8_t* mask,
                  int64_t N, int64_t d, int64_t V, int64_t K, double T, double grad_loss, const double* lse,
                  const int64_t* vrows, int64_t nv_rows, int threads, double* out) {
    (void)V;
    std::fill(out, out + nv_rows * d, 0.0);
    const int64_t nv = count_valid(t, mask, N, K, T);
    if (nv == 0) return;
    parallel_for(nv_rows, threads, [&](int64_t b, int64_t e) {
        std::vector<double> p(static_cast<size_t>(K));
        for (int64_t r = b; r < e; ++r) {
            const int64_t v = vrows[r];
            const double* wv = W + v * d;
            double* o = out + r * d;
            for (int64_t i = 0; i < N; ++i) {
                const bool has = teacher_row(t + i * K, K, T, p.data());
                if (!row_valid(mask, i, has)) continue;
                double z = 0.0;
                for (int64_t j = 0; j < d; ++j) z += h[i * d + j] * wv[j];
                double s = 0.0;
                for (int64_t k = 0; k < K; ++k)
                    if (idx[i * K + k] == v) s += p[k];
                const double c = grad_loss * T / static_cast<double>(nv) * (std::exp(z / T - lse[i]) - s);
                for (int64_t j = 0; j < d; ++j) o[j] += c * h[i * d + j];
            }
        }
    });
}

// KL + hard-label cross-entropy ("Distillyatsiya i szhatie modeley", ml-book.com,
// section "Kak eto rabotaet: myagkie metki i temperatura": the student's loss mixes
// the KL between the softened distributions with the ordinary cross-entropy on the
// true labels; read as the convex mix):
//   loss = alpha T^2 mean KL_i + (1 - alpha) mean CE_i,  CE_i = lse1_i - z_{i,label_i},
//   lse1 the logsumexp of z at temperature 1, means over the valid rows.
void fklo_forward_mix(const double* h, const double* W, const int32_t* idx, const double* t, const uint8_t* mask,
                      const int32_t* label, int64_t N, int64_t d, int64_t V, int64_t K, double T, double alpha,
                      int threads, double* lse, double* lse1, double* kl, double* ce, uint8_t* valid, double* loss,
                      int64_t* n_valid) {
    parallel_for(N, threads, [&](int64_t b, int64_t e) {
        std::vector<double> z(static_cast<size_t>(V)), p(static_cast<size_t>(K));
        for (int64_t i = b; i < e; ++i) {
            const bool has = teacher_row(t + i * K, K, T, p.data());
            valid[i] = row_valid(mask, i, has) ? 1 : 0;
            forward_row(h + i * d, W, idx + i * K, p.data(), d, V, K, T, z.data(), lse + i, kl + i);
            lse1[i] = lse_row(z.data(), V, 1.0);
            ce[i] = lse1[i] - z[label[i]];
        }
    });
    int64_t nv = 0;
    double skl = 0.0, sce = 0.0;
    for (int64_t i = 0; i < N; ++i) {
        if (valid[i]) {
            ++nv;
            skl += kl[i];
            sce += ce[i];
        }
    }
    *n_valid = nv;
    *loss = nv > 0 ? alpha * T * T * skl / static_cast<double>(nv) + (1.0 - alpha) * sce / static_cast<double>(nv)
                   : 0.0;
}

// dh [N][d], dW [V][d] of the mixture times grad_loss:
//   dz_iv = g valid_i [alpha T (q_iv - s_iv) + (1 - alpha)(q1_iv - [v = label_i])] / N_valid.
void fklo_backward_mix(const double* h, const double* W, const int32_t* idx, const double* t, const uint8_t* mask,
                       const int32_t* label, int64_t N, int64_t d, int64_t V, int64_t K, double T, double alpha,
                       double grad_loss, int threads, double* dh, double* dW) {
    std::fill(dh, dh + N * d, 0.0);
    std::fill(dW, dW + V * d, 0.0);
    const int64_t nv = count_valid(t, mask, N, K, T);
    if (nv == 0) return;
    std::vector<double> dz(static_cast<size_t>(N * V));
    parallel_for(N, threads, [&](int64_t b, int64_t e) {
        std::vector<double> z(static_cast<size_t>(V)), p(static_cast<size_t>(K)), q1(static_cast<size_t>(V));
        for (int64_t i = b; i < e; ++i) {
            const bool has = teacher_row(t + i * K, K, T, p.data());
            const double g = row_valid(mask, i, has) ? grad_loss / static_cast<double>(nv) : 0.0;
            double* dzr = dz.data() + i * V;
            logit_row(h + i * d, W, d, V, z.data());
            dz_row(z.data(), idx + i * K, p.data(), V, K, T, lse_row(z.data(), V, T), g * alpha * T, dzr);
            const double l1 = lse_row(z.data(), V, 1.0);
            for (int64_t v = 0; v < V; ++v) q1[v] = std::exp(z[v] - l1);
            q1[label[i]] -= 1.0;
            for (int64_t v = 0; v < V; ++v) dzr[v] += g * (1.0 - alpha) * q1[v];
            add_dh_row(dzr, W, V, d, dh + i * d);
        }
    });
    parallel_for(V, threads, [&](int64_t b, int64_t e) {
        for (int64_t v = b; v < e; ++v) {
            double* dwv = dW + v * d;
            for (int64_t i = 0; i < N; ++i) {
                const double c = dz[i * V + v];
                for (int64_t j = 0; j < d; ++j) dwv[j] += c * h[i * d + j];
            }
        }
    });
}

// Teacher cache: per row the K largest logits (descending, equal logits by
// ascending id) and their ids; idx [N][K], val [N][K].  The top-100 per position
// of "Effektivnaya distillyatsiya znaniy" (malakhovai.ru, paragraph 2).
void fklo_teacher_topk(const double* h, const double* W, int64_t N, int64_t d, int64_t V, int64_t K, int threads,
                       int64_t* idx, double* val) {
    parallel_for(N, threads, [&](int64_t b, int64_t e) {
        std::vector<double> z(static_cast<size_t>(V));
        std::vector<int64_t> ord(static_cast<size_t>(V));
        for (int64_t i = b; i < e; ++i) {
            logit_row(h + i * d, W, d, V, z.data());
            std::iota(ord.begin(), ord.end(), int64_t(0));
            std::partial_sort(ord.begin(), ord.begin() + K, ord.end(), [&](int64_t a, int64_t c) {
                return z[a] > z[c] || (z[a] == z[c] && a < c);
            });
            for (int64_t k = 0; k < K; ++k) {
                idx[i * K + k] = ord[k];
                val[i * K + k] = z[ord[k]];
            }
        }
    });
}

// lse of every row only.
void fklo_student_lse(const double* h, const double* W, int64_t N, int64_t d, int64_t V, double T, int threads,
                      double* lse) {
    parallel_for(N, threads, [&](int64_t b, int64_t e) {
        std::vector<double> z(static_cast<size_t>(V));
        for (int64_t i = b; i < e; ++i) {
            logit_row(h + i * d, W, d, V, z.data());
            lse[i] = lse_row(z.data(), V, T);
        }
    });
}

}  // extern "C"
