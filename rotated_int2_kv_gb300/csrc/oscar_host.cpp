// Host-side parts of liboscar.so: error reporting, argument validation, byte
// accounting, calibration covariances and the rotation builder
// R = U · (H_d/√d) · P_br.
//
// [OSCAR news] "OSCARの違い": U_Q (keys) is the eigenbasis of the query
// covariance C_Q = (1/N) Σ q_nᵀ q_n, U_S (values) the eigenbasis of the
// score-weighted value covariance C_S = (1/N) VᵀSᵀSV; R = U · H_Had · P_br.
// [Escha log] part 2, fix 3: the calibration-free rotation is the Sylvester
// Hadamard matrix divided by sqrt(head_dim).
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstring>
#include <string>
#include <vector>
#include <algorithm>

#include "oscar_internal.h"

namespace oscar {

static thread_local std::string g_err;

int fail(int code, const char* fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof(buf), fmt, ap);
    va_end(ap);
    g_err = buf;
    return code;
}

void clear_error() { g_err.clear(); }

int validate_config(const oscar_config* cfg) {
    if (!cfg) return fail(OSCAR_ERR_NULL, "cfg is NULL");
    const int d = cfg->head_dim;
    if (d != 64 && d != 128 && d != 256)
        return fail(OSCAR_ERR_ARG, "head_dim must be 64, 128 or 256 (got %d)", d);
    if (cfg->num_kv_heads < 1 || cfg->num_kv_heads > 64)
        return fail(OSCAR_ERR_ARG, "num_kv_heads must be in [1, 64] (got %d)", cfg->num_kv_heads);
    if (cfg->num_q_heads < 1 || cfg->num_q_heads % cfg->num_kv_heads != 0)
        return fail(OSCAR_ERR_ARG, "num_q_heads (%d) must be a positive multiple of num_kv_heads (%d)",
                    cfg->num_q_heads, cfg->num_kv_heads);
    const int g = cfg->num_q_heads / cfg->num_kv_heads;
    if (g > 16) return fail(OSCAR_ERR_ARG, "num_q_heads / num_kv_heads must be <= 16 (got %d)", g);
    const int G = cfg->group_size;
    if (!(G == 32 || G == 64 || G == 128 || G == 256) || G > d)
        return fail(OSCAR_ERR_ARG, "group_size must be 32, 64, 128 or 256 and <= head_dim (got %d)", G);
    if (cfg->sink < 0 || cfg->sink > 4096)
        return fail(OSCAR_ERR_ARG, "sink must be in [0, 4096] (got %d)", cfg->sink);
    if (cfg->recent < 1 || cfg->recent > 4096)
        return fail(OSCAR_ERR_ARG, "recent must be in [1, 4096] (got %d)", cfg->recent);
    if (!(cfg->clip_ratio > 0.0f && cfg->clip_ratio <= 1.0f))
        return fail(OSCAR_ERR_ARG, "clip_ratio must be in (0, 1] (got %g)", (double)cfg->clip_ratio);
    if (cfg->kv_dtype != OSCAR_DTYPE_BF16 && cfg->kv_dtype != OSCAR_DTYPE_F32)
        return fail(OSCAR_ERR_ARG, "kv_dtype must be OSCAR_DTYPE_BF16 or OSCAR_DTYPE_F32");
    if (cfg->q_dtype != OSCAR_DTYPE_BF16 && cfg->q_dtype != OSCAR_DTYPE_F32)
        return fail(OSCAR_ERR_ARG, "q_dtype must be OSCAR_DTYPE_BF16 or OSCAR_DTYPE_F32");
    if (cfg->scale_dtype != OSCAR_SCALE_F16 && cfg->scale_dtype != OSCAR_SCALE_E4M3)
        return fail(OSCAR_ERR_ARG, "scale_dtype must be OSCAR_SCALE_F16 or OSCAR_SCALE_E4M3");
    return OSCAR_OK;
}

int validate_cache(const oscar_config* cfg, const oscar_layer_cache* cache) {
    if (!cache) return fail(OSCAR_ERR_NULL, "cache is NULL");
    if (!cache->records) return fail(OSCAR_ERR_NULL, "cache->records is NULL");
    if (!cache->recent) return fail(OSCAR_ERR_NULL, "cache->recent is NULL");
    if (cfg->sink > 0 && !cache->sink) return fail(OSCAR_ERR_NULL, "cache->sink is NULL");
    if (!cache->rot_k || !cache->rot_v) return fail(OSCAR_ERR_NULL, "cache rotation matrices are NULL");
    if (cache->num_slots < 1) return fail(OSCAR_ERR_ARG, "num_slots must be >= 1");
    if (cache->max_reqs < 1) return fail(OSCAR_ERR_ARG, "max_reqs must be >= 1");
    if (reinterpret_cast<uintptr_t>(cache->records) % 16 != 0)
        return fail(OSCAR_ERR_ARG, "cache->records must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(cache->recent) % 16 != 0 ||
        (cache->sink && reinterpret_cast<uintptr_t>(cache->sink) % 16 != 0))
        return fail(OSCAR_ERR_ARG, "window buffers must be 16-byte aligned");
    if (reinterpret_cast<uintptr_t>(cache->rot_k) % 16 != 0 ||
        reinterpret_cast<uintptr_t>(cache->rot_v) % 16 != 0)
        return fail(OSCAR_ERR_ARG, "rotation matrices must be 16-byte aligned");
    return OSCAR_OK;
}

// ---------------------------------------------------------------------------
// Symmetric eigen-decomposition by cyclic Jacobi rotations (fp64).
// Each plane rotation J(p, q, θ) zeroes a[p][q] of Jᵀ·A·J with
// t = tan θ the smaller root of t² + 2·τ·t − 1 = 0, τ = (a_qq − a_pp)/(2 a_pq);
// V accumulates the product of the rotations, so A_0 = V·diag(a)·Vᵀ.
// Sweeps repeat until one full sweep finds every off-diagonal entry
// negligible against its diagonal pair.
// ---------------------------------------------------------------------------
static bool jacobi_eigen(int n, std::vector<double>& a, std::vector<double>& v,
                         std::vector<double>& w) {
    v.assign((size_t)n * n, 0.0);
    for (int i = 0; i < n; ++i) v[(size_t)i * n + i] = 1.0;
    double scale = 0.0;
    for (double x : a) scale = std::max(scale, std::fabs(x));
    const double eps = 2.220446049250313e-16;
    const double tiny = scale * 1e-300 + 1e-300;
    for (int sweep = 0; sweep < 80; ++sweep) {
        int rotations = 0;
        for (int p = 0; p < n - 1; ++p) {
            for (int q = p + 1; q < n; ++q) {
                const double apq = a[(size_t)p * n + q];
                const double app = a[(size_t)p * n + p];
                const double aqq = a[(size_t)q * n + q];
                if (std::fabs(apq) <= tiny ||
                    std::fabs(apq) <= eps * std::sqrt(std::fabs(app)) * std::sqrt(std::fabs(aqq)))
                    continue;
                ++rotations;
                const double tau = (aqq - app) / (2.0 * apq);
                double t;
                if (std::fabs(tau) > 1e150) t = 0.5 / tau;
                else t = (tau >= 0 ? 1.0 : -1.0) / (std::fabs(tau) + std::sqrt(tau * tau + 1.0));
                const double c = 1.0 / std::sqrt(t * t + 1.0);
                const double s = t * c;
                for (int k = 0; k < n; ++k) {  // columns p, q of A·J
                    const double akp = a[(size_t)k * n + p], akq = a[(size_t)k * n + q];
                    a[(size_t)k * n + p] = c * akp - s * akq;
                    a[(size_t)k * n + q] = s * akp + c * akq;
                }
                for (int k = 0; k < n; ++k) {  // rows p, q of Jᵀ·(A·J)
                    const double apk = a[(size_t)p * n + k], aqk = a[(size_t)q * n + k];
                    a[(size_t)p * n + k] = c * apk - s * aqk;
                    a[(size_t)q * n + k] = s * apk + c * aqk;
                }
                a[(size_t)p * n + q] = 0.0;
                a[(size_t)q * n + p] = 0.0;
                for (int k = 0; k < n; ++k) {  // V·J
                    const double vkp = v[(size_t)k * n + p], vkq = v[(size_t)k * n + q];
                    v[(size_t)k * n + p] = c * vkp - s * vkq;
                    v[(size_t)k * n + q] = s * vkp + c * vkq;
                }
            }
        }
        if (rotations == 0) {
            w.resize(n);
            for (int i = 0; i < n; ++i) w[i] = a[(size_t)i * n + i];
            return true;
        }
    }
    return false;
}

static int bitrev(int j, int nbits) {
    int r = 0;
    for (int b = 0; b < nbits; ++b)
        if (j & (1 << b)) r |= 1 << (nbits - 1 - b);
    return r;
}

static int popcount(unsigned x) {
    int c = 0;
    while (x) { c += x & 1u; x >>= 1; }
    return c;
}

}  // namespace oscar

using namespace oscar;

extern "C" {

const char* oscar_version(void) { return "oscar-gb300 0.1 (sm_103a)"; }

const char* oscar_last_error(void) { return g_err.c_str(); }

int oscar_record_bytes(const oscar_config* cfg, int64_t* out) {
    clear_error();
    int rc = validate_config(cfg);
    if (rc) return rc;
    if (!out) return fail(OSCAR_ERR_NULL, "out is NULL");
    *out = record_layout(cfg->head_dim, cfg->group_size, cfg->scale_dtype).bytes;
    return OSCAR_OK;
}

int oscar_slot_bytes(const oscar_config* cfg, int64_t* out) {
    clear_error();
    int rc = validate_config(cfg);
    if (rc) return rc;
    if (!out) return fail(OSCAR_ERR_NULL, "out is NULL");
    *out = slot_bytes(record_layout(cfg->head_dim, cfg->group_size, cfg->scale_dtype), cfg->num_kv_heads);
    return OSCAR_OK;
}

int oscar_cache_bytes_per_token(const oscar_config* cfg, int64_t* int2_bytes, int64_t* bf16_bytes) {
    clear_error();
    int rc = validate_config(cfg);
    if (rc) return rc;
    if (!int2_bytes || !bf16_bytes) return fail(OSCAR_ERR_NULL, "output pointer is NULL");
    *int2_bytes = slot_bytes(record_layout(cfg->head_dim, cfg->group_size, cfg->scale_dtype), cfg->num_kv_heads);
    *bf16_bytes = (int64_t)cfg->num_kv_heads * 2 * cfg->head_dim * 2;
    return OSCAR_OK;
}

int oscar_covariance(const double* samples, int64_t n, int32_t d, double* cov) {
    clear_error();
    if (!samples || !cov) return fail(OSCAR_ERR_NULL, "samples and cov must be non-NULL");
    if (n < 1 || d < 1 || d > 4096) return fail(OSCAR_ERR_ARG, "need n >= 1 and 1 <= d <= 4096");
    std::vector<double> acc((size_t)d * d, 0.0);
    for (int64_t s = 0; s < n; ++s) {
        const double* x = samples + s * d;
        for (int i = 0; i < d; ++i) {
            const double xi = x[i];
            double* row = acc.data() + (size_t)i * d;
            for (int j = i; j < d; ++j) row[j] += xi * x[j];
        }
    }
    for (int i = 0; i < d; ++i)
        for (int j = i; j < d; ++j) {
            const double c = acc[(size_t)i * d + j] / (double)n;
            cov[(size_t)i * d + j] = c;
            cov[(size_t)j * d + i] = c;
        }
    return OSCAR_OK;
}

int oscar_value_covariance(const double* scores, const double* values, int64_t n_q, int64_t n_k,
                           int32_t d, double* cov) {
    clear_error();
    if (!scores || !values || !cov) return fail(OSCAR_ERR_NULL, "scores, values and cov must be non-NULL");
    if (n_q < 1 || n_k < 1 || d < 1 || d > 4096) return fail(OSCAR_ERR_ARG, "need n_q, n_k >= 1 and 1 <= d <= 4096");
    // rows of S·V are the score-weighted values; C_S is their second moment over n_q.
    std::vector<double> sv((size_t)n_q * d, 0.0);
    for (int64_t a = 0; a < n_q; ++a) {
        double* out = sv.data() + (size_t)a * d;
        for (int64_t t = 0; t < n_k; ++t) {
            const double s = scores[a * n_k + t];
            if (s == 0.0) continue;
            const double* vr = values + t * d;
            for (int i = 0; i < d; ++i) out[i] += s * vr[i];
        }
    }
    return oscar_covariance(sv.data(), n_q, d, cov);
}

int oscar_build_rotation(const double* cov, int32_t d, int32_t use_bitrev, float* R_f32,
                         double* R_f64, double* eigvals) {
    return oscar_build_rotation_ex(cov, d, use_bitrev, d, R_f32, R_f64, eigvals);
}

int oscar_build_rotation_ex(const double* cov, int32_t d, int32_t use_bitrev, int32_t hadamard_block,
                            float* R_f32, double* R_f64, double* eigvals) {
    clear_error();
    if (!R_f32) return fail(OSCAR_ERR_NULL, "R_f32 is NULL");
    if (d < 2 || d > 256 || (d & (d - 1)) != 0) return fail(OSCAR_ERR_ARG, "d must be a power of two in [2, 256]");
    if (hadamard_block < 1 || hadamard_block > d || (hadamard_block & (hadamard_block - 1)) != 0)
        return fail(OSCAR_ERR_ARG, "hadamard_block must be a power of two in [1, d]");
    const int n = d;
    std::vector<double> U((size_t)n * n, 0.0), w(n, 1.0);
    if (cov) {
        std::vector<double> a(cov, cov + (size_t)n * n);
        for (int i = 0; i < n; ++i)
            for (int j = i + 1; j < n; ++j) {
                const double m = 0.5 * (a[(size_t)i * n + j] + a[(size_t)j * n + i]);
                if (!std::isfinite(m)) return fail(OSCAR_ERR_ARG, "covariance has a non-finite entry");
                a[(size_t)i * n + j] = m;
                a[(size_t)j * n + i] = m;
            }
        std::vector<double> V, ev;
        if (!jacobi_eigen(n, a, V, ev)) return fail(OSCAR_ERR_NUMERIC, "Jacobi eigensolver did not converge");
        std::vector<int> order(n);
        for (int i = 0; i < n; ++i) order[i] = i;
        std::stable_sort(order.begin(), order.end(), [&](int x, int y) { return ev[x] > ev[y]; });
        for (int jc = 0; jc < n; ++jc) {
            const int src = order[jc];
            w[jc] = ev[src];
            int imax = 0;
            double vmax = -1.0;
            for (int i = 0; i < n; ++i) {
                const double m = std::fabs(V[(size_t)i * n + src]);
                if (m > vmax) { vmax = m; imax = i; }
            }
            const double sgn = V[(size_t)imax * n + src] < 0 ? -1.0 : 1.0;
            for (int i = 0; i < n; ++i) U[(size_t)i * n + jc] = sgn * V[(size_t)i * n + src];
        }
    } else {
        for (int i = 0; i < n; ++i) U[(size_t)i * n + i] = 1.0;
    }
    // M = U · H with H block-diagonal: blocks of B = hadamard_block channels,
    // H[k][j] = (-1)^popcount(k & j)/√B when k and j share a block (Sylvester
    // closed form within the block), else 0.  B = d is the full Hadamard.
    const int B = hadamard_block;
    const double inv = 1.0 / std::sqrt((double)B);
    std::vector<double> M((size_t)n * n, 0.0);
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j) {
            double acc = 0.0;
            const int k0 = j / B * B;
            for (int k = k0; k < k0 + B; ++k) {
                const double u = U[(size_t)i * n + k];
                acc += (popcount((unsigned)(k & j & (B - 1))) & 1) ? -u : u;
            }
            M[(size_t)i * n + j] = acc * inv;
        }
    int nbits = 0;
    while ((1 << nbits) < n) ++nbits;
    for (int i = 0; i < n; ++i)
        for (int j = 0; j < n; ++j) {
            const int src = use_bitrev ? bitrev(j, nbits) : j;
            const double r = M[(size_t)i * n + src];
            if (R_f64) R_f64[(size_t)i * n + j] = r;
            R_f32[(size_t)i * n + j] = (float)r;
        }
    if (eigvals)
        for (int i = 0; i < n; ++i) eigvals[i] = cov ? w[i] : 1.0;
    return OSCAR_OK;
}

}  // extern "C"
