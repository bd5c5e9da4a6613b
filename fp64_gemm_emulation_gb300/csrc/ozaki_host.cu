// ozaki_host.cu -- the C ABI of libozaki: argument checks, parameters, workspace,
// and the launch sequence of the Ozaki Scheme II path.
//
// Parameters follow [Ozaki II]: the moduli (section 6: 2 <= m_t <= 256, pairwise
// coprime; the greedy descending list from 256 is used), M = prod m_t, M_t = M / m_t,
// y_t = M_t^{-1} mod m_t (section 4), and k_A = k_B = the largest k with
// q 2^(2k) <= M/2 - 1 (section 5), computed exactly on multi-limb integers.
#include <atomic>
#include <cstdio>
#include <cstring>

#include "oz_internal.h"

namespace oz {
namespace {

// ---------------------------------------------------------------- small big-integer
constexpr int kBigLimbs = 8;  // 256 bits: M < 2^160, q 4^k < 2^162
struct Big {
  uint32_t w[kBigLimbs];
};

Big big_from(uint64_t v) {
  Big b{};
  b.w[0] = static_cast<uint32_t>(v);
  b.w[1] = static_cast<uint32_t>(v >> 32);
  return b;
}

Big big_mul_small(const Big& a, uint32_t m) {
  Big r{};
  uint64_t carry = 0;
  for (int i = 0; i < kBigLimbs; ++i) {
    const uint64_t v = static_cast<uint64_t>(a.w[i]) * m + carry;
    r.w[i] = static_cast<uint32_t>(v);
    carry = v >> 32;
  }
  return r;
}

Big big_div_small(const Big& a, uint32_t m, uint32_t* rem) {
  Big q{};
  uint64_t r = 0;
  for (int i = kBigLimbs - 1; i >= 0; --i) {
    const uint64_t cur = (r << 32) | a.w[i];
    q.w[i] = static_cast<uint32_t>(cur / m);
    r = cur % m;
  }
  if (rem) *rem = static_cast<uint32_t>(r);
  return q;
}

int big_cmp(const Big& a, const Big& b) {
  for (int i = kBigLimbs - 1; i >= 0; --i)
    if (a.w[i] != b.w[i]) return a.w[i] < b.w[i] ? -1 : 1;
  return 0;
}

Big big_sub_small(const Big& a, uint32_t v) {
  Big r = a;
  uint64_t borrow = v;
  for (int i = 0; i < kBigLimbs && borrow; ++i) {
    const uint64_t cur = r.w[i];
    r.w[i] = static_cast<uint32_t>(cur - borrow);
    borrow = cur < borrow ? 1 : 0;
  }
  return r;
}

// The greedy descending pairwise-coprime list starting at 256.
int greedy_moduli(int s, int* out) {
  int count = 0;
  for (int cand = 256; cand >= 2 && count < s; --cand) {
    bool ok = true;
    for (int i = 0; i < count && ok; ++i) {
      int a = cand, b = out[i];
      while (b) {
        const int t = a % b;
        a = b;
        b = t;
      }
      ok = (a == 1);
    }
    if (ok) out[count++] = cand;
  }
  return count;
}

struct Params {
  int s;
  int mod[kMaxModuli];
  Big M;
  Big P[kMaxModuli];  // M_t * y_t
  int y[kMaxModuli];
};

int make_params(int s, Params* p) {
  if (s < 1 || s > kMaxModuli) return OZ_EINVAL;
  p->s = s;
  if (greedy_moduli(s, p->mod) != s) return OZ_EINVAL;
  p->M = big_from(1);
  for (int t = 0; t < s; ++t) p->M = big_mul_small(p->M, static_cast<uint32_t>(p->mod[t]));
  for (int t = 0; t < s; ++t) {
    const uint32_t m = static_cast<uint32_t>(p->mod[t]);
    uint32_t unused;
    const Big Mt = big_div_small(p->M, m, &unused);
    uint32_t Mt_mod;
    big_div_small(Mt, m, &Mt_mod);
    int y = -1;
    for (uint32_t c = 1; c < m; ++c)
      if ((static_cast<uint64_t>(Mt_mod) * c) % m == 1) {
        y = static_cast<int>(c);
        break;
      }
    if (y < 0) return OZ_EINVAL;
    p->y[t] = y;
    p->P[t] = big_mul_small(Mt, static_cast<uint32_t>(y));
  }
  return OZ_OK;
}

// Largest k >= 0 with 2 q 4^k <= M - 2; -1 if none.
int choose_k(const Big& M, long long q) {
  if (q < 1) return -1;
  const Big lim = big_sub_small(M, 2);
  Big t = big_mul_small(big_from(static_cast<uint64_t>(q)), 2);
  if (big_cmp(t, lim) > 0) return -1;
  int k = 0;
  while (true) {
    const Big t4 = big_mul_small(t, 4);
    if (big_cmp(t4, lim) > 0) break;
    t = t4;
    ++k;
  }
  return k;
}

}  // namespace

int fill_split_consts(int s, long long k_inner, SplitConsts* out) {
  Params p;
  int rc = make_params(s, &p);
  if (rc) return rc;
  const int k = choose_k(p.M, k_inner);
  if (k < 1) return OZ_ERANGE;
  std::memset(out, 0, sizeof(*out));
  out->s = s;
  out->kA = k;
  out->shift_ok = 1;
  for (int t = 0; t < s; ++t) {
    const uint32_t m = static_cast<uint32_t>(p.mod[t]);
    if ((static_cast<uint64_t>(m) << 22) <= (1ull << 26)) out->shift_ok = 0;
    out->mod[t] = p.mod[t];
    out->c16[t] = (1u << 16) % m;
    out->c32[t] = static_cast<uint32_t>((1ull << 32) % m);
    out->c48[t] = static_cast<uint32_t>((1ull << 48) % m);
    out->c64[t] = static_cast<uint32_t>((static_cast<uint64_t>(out->c48[t]) * out->c16[t]) % m);
    out->c80[t] = static_cast<uint32_t>((static_cast<uint64_t>(out->c64[t]) * out->c16[t]) % m);
    out->magic[t] = static_cast<uint32_t>(((1ull << 39) + m - 1) / m);
    out->offs[t] = (m << 22) + (m >> 1);
    out->fbase[t] = 0x4B000080u - (m >> 1);
    out->f13[t] = static_cast<float>((1u << 13) % m);
    out->f26[t] = static_cast<float>((1u << 26) % m);
    out->f39[t] = static_cast<float>((1ull << 39) % m);
    out->finv[t] = 1.0f / static_cast<float>(m);  // correctly rounded FP32 division
    out->fmod[t] = static_cast<float>(m);
  }
  out->limb13_ok = (s >= 1 && p.mod[0] == 256) ? 1 : 0;
  for (int t = 1; t < s; ++t)
    if (p.mod[t] % 2 == 0 || p.mod[t] <= 128 || p.mod[t] >= 256) out->limb13_ok = 0;
  return OZ_OK;
}

int fill_crt_consts(int s, long long k_inner, CrtConsts* out) {
  Params p;
  int rc = make_params(s, &p);
  if (rc) return rc;
  const int k = choose_k(p.M, k_inner);
  if (k < 1) return OZ_ERANGE;
  std::memset(out, 0, sizeof(*out));
  out->s = s;
  out->kA = k;
  for (int l = kLimbs; l < kBigLimbs; ++l)
    if (p.M.w[l]) return OZ_EINVAL;  // cannot happen for <= 20 moduli <= 256
  uint32_t unused;
  const Big half = big_div_small(p.M, 2, &unused);
  for (int l = 0; l < kLimbs; ++l) {
    out->M[l] = p.M.w[l];
    out->halfM[l] = half.w[l];
  }
  int mbits = 0;
  for (int l = kLimbs - 1; l >= 0 && !mbits; --l)
    if (p.M.w[l]) mbits = 32 * l + (32 - __builtin_clz(p.M.w[l]));
  out->n16 = (mbits + 15) / 16;
  if (out->n16 > kHalfLimbs) return OZ_EINVAL;  // cannot happen for <= 20 moduli <= 256
  for (int t = 0; t < s; ++t) {
    out->mod[t] = p.mod[t];
    for (int l = 0; l < kLimbs; ++l) out->P[t][l] = p.P[t].w[l];
    for (int l = 0; l < kHalfLimbs; ++l) {  // bits [16 l, 16 l + 16) of P_t
      const uint32_t half = (p.P[t].w[l >> 1] >> (16 * (l & 1))) & 0xFFFFu;
      out->Pd[t >> 1][l] |= half << (16 * (t & 1));
    }
  }
  return OZ_OK;
}

int half_range_log2(int s) {
  Params p;
  if (make_params(s, &p)) return -1;
  const Big lim = big_sub_small(p.M, 2);  // 2^(L+1) <= M - 2 < 2^(L+2)
  for (int i = kBigLimbs - 1; i >= 0; --i)
    if (lim.w[i]) return 32 * i + (31 - __builtin_clz(lim.w[i])) - 1;
  return -1;
}

}  // namespace oz

using namespace oz;

namespace {

struct Layout {
  int mp, np, kp;
  size_t off_rowexp, off_colexp, off_A, off_B, off_C, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

Layout make_layout(int m, int n, int k, int s) {
  Layout L;
  L.mp = static_cast<int>(roundup(m, kPadM));
  L.np = static_cast<int>(roundup(n, kPadN));
  L.kp = static_cast<int>(roundup(k, kPadK));
  size_t off = 0;
  L.off_rowexp = off;
  off = align256(off + sizeof(int32_t) * static_cast<size_t>(m));
  L.off_colexp = off;
  off = align256(off + sizeof(int32_t) * static_cast<size_t>(n));
  L.off_A = off;
  off = align256(off + sizeof(uint16_t) * static_cast<size_t>(s) * L.mp * L.kp);
  L.off_B = off;
  off = align256(off + sizeof(uint16_t) * static_cast<size_t>(s) * L.np * L.kp);
  L.off_C = off;
  off = align256(off + static_cast<size_t>(s) * L.np * L.mp);
  L.total = off;
  return L;
}

int check_dims(int m, int n, int k, int lda, int ldb, int ldc) {
  if (m < 0 || n < 0 || k < 0) return OZ_EINVAL;
  if (lda < (m > 1 ? m : 1) || ldb < (k > 1 ? k : 1) || ldc < (m > 1 ? m : 1)) return OZ_EINVAL;
  return OZ_OK;
}

int cuda_rc(cudaError_t e) { return e == cudaSuccess ? OZ_OK : OZ_ECUDA; }

// The allocating entry points draw their workspace from the device's default
// stream-ordered memory pool.  Raise its release threshold once per device so the
// pool keeps the memory between calls instead of unmapping it at every
// synchronisation (repeated calls then allocate in microseconds).
void keep_default_pool_cached() {
  static std::atomic<bool> done[64] = {};  // several host threads may call at once
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || done[dev].load(std::memory_order_acquire))
    return;
  cudaMemPool_t pool;
  if (cudaDeviceGetDefaultMemPool(&pool, dev) == cudaSuccess) {
    uint64_t threshold = ~0ull;
    cudaMemPoolSetAttribute(pool, cudaMemPoolAttrReleaseThreshold, &threshold);  // idempotent
  }
  cudaGetLastError();
  done[dev].store(true, std::memory_order_release);
}

// A dimension cut into up to kMax blocks whose sizes are multiples of 256 (but the last).
struct Blocks {
  static constexpr int kMax = 8;
  int count;
  int start[kMax], size[kMax];
};

Blocks make_blocks(int d, int want) {
  Blocks b{};
  if (want < 1) want = 1;
  if (want > Blocks::kMax) want = Blocks::kMax;
  const int bs = static_cast<int>(roundup((d + want - 1) / want, 256));
  for (int s0 = 0; s0 < d && b.count < Blocks::kMax; s0 += bs) {
    b.start[b.count] = s0;
    b.size[b.count] = (d - s0 < bs) ? d - s0 : bs;
    ++b.count;
  }
  return b;
}

GemmConsts make_gemm_consts(const SplitConsts& sc) {
  GemmConsts g{};
  g.s = sc.s;
  for (int t = 0; t < sc.s; ++t) {
    g.modf[t] = static_cast<float>(sc.mod[t]);
    g.invf[t] = static_cast<float>(1.0 / sc.mod[t]);
  }
  return g;
}

bool valid_scaling(int scaling) {
  return scaling == OZ_SCALE_UNIFORM || scaling == OZ_SCALE_FAST || scaling == OZ_SCALE_ACCU;
}

// The inner dimension whose k_A the split and the CRT use: the uniform estimate bounds
// c_max by q 2^(k_A + k_B); fast and accu bound it by 2^(2 kappa), the k_A of q = 1.
long long scaling_q(int scaling, long long k) { return scaling == OZ_SCALE_UNIFORM ? k : 1; }

// OS II-accu: the largest b in [0, 7] with q 4^b <= 2^24; -1 when q > 2^24.
int accu_bits(long long q) {
  if (q < 1 || q > (1LL << 24)) return -1;
  int b = 0;
  while (b < 7 && (q << (2 * b + 2)) <= (1LL << 24)) ++b;
  return b;
}

// Workspace of the exponent step (scaling modes other than uniform).
struct ExpLayout {
  size_t off_S_row, off_S_col;           // fast: uint64 [m], [n]
  size_t off_Ahat, off_Bhat, off_maxes;  // accu: bf16 [Mp][Kp], [Np][Kp]; uint32 [Mp + Np]
  size_t total;
};

ExpLayout make_exp_layout(int m, int n, int k, int scaling) {
  ExpLayout E{};
  const size_t mp = static_cast<size_t>(roundup(m, kPadM)), np = static_cast<size_t>(roundup(n, kPadN)),
               kp = static_cast<size_t>(roundup(k, kPadK));
  size_t off = 0;
  if (scaling == OZ_SCALE_FAST) {
    E.off_S_row = off;
    off = align256(off + sizeof(unsigned long long) * static_cast<size_t>(m));
    E.off_S_col = off;
    off = align256(off + sizeof(unsigned long long) * static_cast<size_t>(n));
  } else if (scaling == OZ_SCALE_ACCU) {
    E.off_Ahat = off;
    off = align256(off + sizeof(uint16_t) * mp * kp);
    E.off_Bhat = off;
    off = align256(off + sizeof(uint16_t) * np * kp);
    E.off_maxes = off;
    off = align256(off + sizeof(uint32_t) * (mp + np));
  }
  E.total = off;
  return E;
}

// Whole-call workspace: the exponent step's scratch lives where C_res will go (it is
// consumed before the split, and C_res is written only by the GEMM after it).
size_t total_bytes_ex(const Layout& L, int m, int n, int k, int scaling) {
  const size_t e = L.off_C + make_exp_layout(m, n, k, scaling).total;
  return e > L.total ? align256(e) : L.total;
}

}  // namespace

extern "C" {

int ozaki2_moduli(int num_moduli, int* moduli_out) {
  if (!moduli_out || num_moduli < 1 || num_moduli > OZ_MAX_MODULI) return OZ_EINVAL;
  return oz::greedy_moduli(num_moduli, moduli_out) == num_moduli ? OZ_OK : OZ_EINVAL;
}

int ozaki2_choose_k(int num_moduli, long long k_inner, int* k_out) {
  if (!k_out || k_inner < 1) return OZ_EINVAL;
  Params p;
  const int rc = make_params(num_moduli, &p);
  if (rc) return rc;
  const int k = oz::choose_k(p.M, k_inner);
  if (k < 1) return OZ_ERANGE;
  *k_out = k;
  return OZ_OK;
}

int ozaki2_plane_dims(int m, int n, int k, int* mp, int* np, int* kp) {
  if (m < 0 || n < 0 || k < 0 || !mp || !np || !kp) return OZ_EINVAL;
  *mp = static_cast<int>(roundup(m, kPadM));
  *np = static_cast<int>(roundup(n, kPadN));
  *kp = static_cast<int>(roundup(k, kPadK));
  return OZ_OK;
}

size_t ozaki2_workspace_bytes(int m, int n, int k, int num_moduli) {
  if (m < 0 || n < 0 || k < 0 || num_moduli < OZ_MIN_MODULI || num_moduli > OZ_MAX_MODULI) return 0;
  return make_layout(m, n, k, num_moduli).total;
}

int ozaki2_exponents(int m, int n, int k, const double* A, int lda, const double* B, int ldb, int32_t* rowexp,
                     int32_t* colexp, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 0) return OZ_EINVAL;
  if ((A && (lda < (m > 1 ? m : 1) || !rowexp)) || (B && (ldb < (k > 1 ? k : 1) || !colexp))) return OZ_EINVAL;
  return cuda_rc(launch_exponents(m, n, k, A, lda, B, ldb, rowexp, colexp, stream));
}

int ozaki2_scaling_k(int num_moduli, long long k_inner, int scaling, int* k_out) {
  if (!valid_scaling(scaling)) return OZ_EINVAL;
  if (scaling == OZ_SCALE_ACCU && accu_bits(k_inner) < 0) return OZ_EINVAL;
  if (!k_out || k_inner < 1) return OZ_EINVAL;
  return ozaki2_choose_k(num_moduli, scaling_q(scaling, k_inner), k_out);
}

size_t ozaki2_exponents_workspace_bytes(int m, int n, int k, int scaling) {
  if (m < 0 || n < 0 || k < 0 || !valid_scaling(scaling)) return 0;
  return make_exp_layout(m, n, k, scaling).total;
}

int ozaki2_exponents_ex(int m, int n, int k, const double* A, int lda, const double* B, int ldb, int num_moduli,
                        int scaling, int32_t* rowexp, int32_t* colexp, void* workspace, size_t ws_bytes,
                        cudaStream_t stream) {
  if (!valid_scaling(scaling) || num_moduli < OZ_MIN_MODULI || num_moduli > OZ_MAX_MODULI) return OZ_EINVAL;
  if (scaling == OZ_SCALE_UNIFORM) return ozaki2_exponents(m, n, k, A, lda, B, ldb, rowexp, colexp, stream);
  if (m < 0 || n < 0 || k < 0) return OZ_EINVAL;
  if ((A && (lda < (m > 1 ? m : 1) || !rowexp)) || (B && (ldb < (k > 1 ? k : 1) || !colexp))) return OZ_EINVAL;
  if (scaling == OZ_SCALE_ACCU && (!A || !B || (k > 0 && accu_bits(k) < 0))) return OZ_EINVAL;
  const ExpLayout E = make_exp_layout(m, n, k, scaling);
  if (E.total && (!workspace || ws_bytes < E.total || (reinterpret_cast<uintptr_t>(workspace) & 255)))
    return OZ_ENOMEM;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  if (scaling == OZ_SCALE_FAST)
    return cuda_rc(launch_norm_exponents(m, n, k, A, lda, B, ldb, rowexp, colexp,
                                         reinterpret_cast<unsigned long long*>(ws + E.off_S_row),
                                         reinterpret_cast<unsigned long long*>(ws + E.off_S_col), stream));
  // OS II-accu: maxima exponents, rounded-up magnitudes, their exact product's row and
  // column maxima, then the exponents of the scaling.
  int rc = cuda_rc(launch_exponents(m, n, k, A, lda, B, ldb, rowexp, colexp, stream));
  if (rc || k == 0 || m == 0 || n == 0) return rc;
  Params p;
  if ((rc = make_params(num_moduli, &p))) return rc;
  const int kappa = oz::choose_k(p.M, 1);
  const int L = half_range_log2(num_moduli);
  const int b = accu_bits(k);
  if (kappa < 1 || L < 0 || b < 0) return OZ_EINVAL;
  const int mp = static_cast<int>(roundup(m, kPadM)), np = static_cast<int>(roundup(n, kPadN)),
            kp = static_cast<int>(roundup(k, kPadK));
  uint16_t* Ahat = reinterpret_cast<uint16_t*>(ws + E.off_Ahat);
  uint16_t* Bhat = reinterpret_cast<uint16_t*>(ws + E.off_Bhat);
  uint32_t* maxes = reinterpret_cast<uint32_t*>(ws + E.off_maxes);
  if ((rc = cuda_rc(launch_magnitudes(m, k, A, 1, lda, rowexp, b, Ahat, mp, kp, stream)))) return rc;
  if ((rc = cuda_rc(launch_magnitudes(n, k, B, ldb, 1, colexp, b, Bhat, np, kp, stream)))) return rc;
  if ((rc = launch_bound_gemm(mp, np, kp, Ahat, Bhat, maxes, stream))) return rc;
  if ((rc = cuda_rc(launch_accu_finalize(m, rowexp, maxes, L, kappa, b, stream)))) return rc;
  return cuda_rc(launch_accu_finalize(n, colexp, maxes + mp, L, kappa, b, stream));
}

int ozaki2_split(int m, int n, int k, const double* A, int lda, const double* B, int ldb, int num_moduli,
                 const int32_t* rowexp, const int32_t* colexp, uint16_t* A_planes, uint16_t* B_planes,
                 cudaStream_t stream) {
  return ozaki2_split_ex(m, n, k, A, lda, B, ldb, num_moduli, OZ_SCALE_UNIFORM, rowexp, colexp, A_planes, B_planes,
                         stream);
}

int ozaki2_split_ex(int m, int n, int k, const double* A, int lda, const double* B, int ldb, int num_moduli,
                    int scaling, const int32_t* rowexp, const int32_t* colexp, uint16_t* A_planes,
                    uint16_t* B_planes, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 1 || !valid_scaling(scaling)) return OZ_EINVAL;
  if ((A && (lda < (m > 1 ? m : 1) || !rowexp || !A_planes)) || (B && (ldb < (k > 1 ? k : 1) || !colexp || !B_planes)))
    return OZ_EINVAL;
  if (num_moduli < OZ_MIN_MODULI || num_moduli > OZ_MAX_MODULI) return OZ_EINVAL;
  SplitConsts sc;
  int rc = fill_split_consts(num_moduli, scaling_q(scaling, k), &sc);
  if (rc) return rc;
  const int mp = static_cast<int>(roundup(m, kPadM)), np = static_cast<int>(roundup(n, kPadN)),
            kp = static_cast<int>(roundup(k, kPadK));
  if (A && m > 0) {
    rc = cuda_rc(launch_split(m, k, A, 1, lda, rowexp, sc, A_planes, mp, kp, stream));
    if (rc) return rc;
  }
  if (B && n > 0) {
    rc = cuda_rc(launch_split(n, k, B, ldb, 1, colexp, sc, B_planes, np, kp, stream));
    if (rc) return rc;
  }
  return OZ_OK;
}

// Longest padded k for which B's exponents and split take one DRAM pass.
constexpr int kFusedMaxKp = 16384;

int ozaki2_scale_split(int m, int n, int k, const double* A, int lda, const double* B, int ldb, int num_moduli,
                       int32_t* rowexp, int32_t* colexp, uint16_t* A_planes, uint16_t* B_planes,
                       cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 1) return OZ_EINVAL;
  if ((A && (lda < (m > 1 ? m : 1) || !rowexp || !A_planes)) || (B && (ldb < (k > 1 ? k : 1) || !colexp || !B_planes)))
    return OZ_EINVAL;
  if (num_moduli < OZ_MIN_MODULI || num_moduli > OZ_MAX_MODULI) return OZ_EINVAL;
  SplitConsts sc;
  int rc = fill_split_consts(num_moduli, k, &sc);
  if (rc) return rc;
  const int np = static_cast<int>(roundup(n, kPadN)), kp = static_cast<int>(roundup(k, kPadK));
  // B: one DRAM pass (each column's maximum, then its residues, the second read from L2) while
  // a column fits in L2 many times over (Kp <= 16384: the resident blocks hold about 40 MB of
  // columns); above that, the exponent pass and the split.  A: the exponent pass, then the split.
  if (B && n > 0) {
    if (kp <= kFusedMaxKp) {
      rc = cuda_rc(launch_split_fused_kcontig(n, k, B, ldb, sc, colexp, B_planes, np, kp, stream));
    } else {
      rc = ozaki2_exponents(0, n, k, nullptr, 1, B, ldb, nullptr, colexp, stream);
      if (!rc) rc = ozaki2_split(0, n, k, nullptr, 1, B, ldb, num_moduli, nullptr, colexp, nullptr, B_planes, stream);
    }
    if (rc) return rc;
  }
  if (A && m > 0) {
    if ((rc = ozaki2_exponents(m, 0, k, A, lda, nullptr, 1, rowexp, nullptr, stream))) return rc;
    rc = ozaki2_split(m, 0, k, A, lda, nullptr, 1, num_moduli, rowexp, nullptr, A_planes, nullptr, stream);
  }
  return rc;
}

int ozaki2_residue_gemm(int m, int n, int k, int num_moduli, const uint16_t* A_planes, const uint16_t* B_planes,
                        uint8_t* C_res, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 1 || !A_planes || !B_planes || !C_res) return OZ_EINVAL;
  if (num_moduli < OZ_MIN_MODULI || num_moduli > OZ_MAX_MODULI) return OZ_EINVAL;
  if (m == 0 || n == 0) return OZ_OK;
  SplitConsts sc;  // only the moduli are used: no dependence on k_A or the scaling mode
  const int rc = fill_split_consts(num_moduli, 1, &sc);
  if (rc) return rc;
  return launch_residue_gemm(static_cast<int>(roundup(m, kPadM)), static_cast<int>(roundup(n, kPadN)),
                             static_cast<int>(roundup(k, kPadK)), make_gemm_consts(sc), A_planes, B_planes, C_res,
                             stream);
}

int ozaki2_crt(int m, int n, int k, int num_moduli, const uint8_t* C_res, const int32_t* rowexp,
               const int32_t* colexp, double* C, int ldc, cudaStream_t stream) {
  return ozaki2_crt_ex(m, n, k, num_moduli, OZ_SCALE_UNIFORM, C_res, rowexp, colexp, C, ldc, stream);
}

int ozaki2_crt_ex(int m, int n, int k, int num_moduli, int scaling, const uint8_t* C_res, const int32_t* rowexp,
                  const int32_t* colexp, double* C, int ldc, cudaStream_t stream) {
  if (m < 0 || n < 0 || k < 1 || !C_res || !rowexp || !colexp || !C || ldc < (m > 1 ? m : 1)) return OZ_EINVAL;
  if (num_moduli < OZ_MIN_MODULI || num_moduli > OZ_MAX_MODULI || !valid_scaling(scaling)) return OZ_EINVAL;
  CrtConsts cc;
  const int rc = fill_crt_consts(num_moduli, scaling_q(scaling, k), &cc);
  if (rc) return rc;
  return cuda_rc(launch_crt(m, n, static_cast<int>(roundup(m, kPadM)), static_cast<int>(roundup(n, kPadN)), cc,
                            C_res, rowexp, colexp, C, ldc, stream));
}

int ozaki2_dgemm_ws(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc,
                    int num_moduli, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_dims(m, n, k, lda, ldb, ldc);
  if (rc) return rc;
  if (num_moduli < OZ_MIN_MODULI || num_moduli > OZ_MAX_MODULI) return OZ_EINVAL;
  if (m == 0 || n == 0) return OZ_OK;
  if (!C) return OZ_EINVAL;
  if (k == 0) return cuda_rc(launch_fill_zero(m, n, C, ldc, stream));
  if (!A || !B) return OZ_EINVAL;
  {
    int kA;
    rc = ozaki2_choose_k(num_moduli, k, &kA);
    if (rc) return rc;
  }
  const Layout L = make_layout(m, n, k, num_moduli);
  if (!workspace || ws_bytes < L.total || (reinterpret_cast<uintptr_t>(workspace) & 255)) return OZ_ENOMEM;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* rowexp = reinterpret_cast<int32_t*>(ws + L.off_rowexp);
  int32_t* colexp = reinterpret_cast<int32_t*>(ws + L.off_colexp);
  uint16_t* Ap = reinterpret_cast<uint16_t*>(ws + L.off_A);
  uint16_t* Bp = reinterpret_cast<uint16_t*>(ws + L.off_B);
  uint8_t* Cr = ws + L.off_C;
  if ((rc = ozaki2_scale_split(m, n, k, A, lda, B, ldb, num_moduli, rowexp, colexp, Ap, Bp, stream))) return rc;
  if ((rc = ozaki2_residue_gemm(m, n, k, num_moduli, Ap, Bp, Cr, stream))) return rc;
  return ozaki2_crt(m, n, k, num_moduli, Cr, rowexp, colexp, C, ldc, stream);
}

size_t ozaki2_workspace_bytes_ex(int m, int n, int k, int num_moduli, int scaling) {
  if (m < 0 || n < 0 || k < 0 || num_moduli < OZ_MIN_MODULI || num_moduli > OZ_MAX_MODULI || !valid_scaling(scaling))
    return 0;
  return total_bytes_ex(make_layout(m, n, k, num_moduli), m, n, k, scaling);
}

int ozaki2_dgemm_ex_ws(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc,
                       int num_moduli, int scaling, void* workspace, size_t ws_bytes, cudaStream_t stream) {
  int rc = check_dims(m, n, k, lda, ldb, ldc);
  if (rc) return rc;
  if (num_moduli < OZ_MIN_MODULI || num_moduli > OZ_MAX_MODULI || !valid_scaling(scaling)) return OZ_EINVAL;
  if (m == 0 || n == 0) return OZ_OK;
  if (!C) return OZ_EINVAL;
  if (k == 0) return cuda_rc(launch_fill_zero(m, n, C, ldc, stream));
  if (!A || !B) return OZ_EINVAL;
  {
    int kA;
    if ((rc = ozaki2_scaling_k(num_moduli, k, scaling, &kA))) return rc;
  }
  const Layout L = make_layout(m, n, k, num_moduli);
  const size_t total = total_bytes_ex(L, m, n, k, scaling);
  if (!workspace || ws_bytes < total || (reinterpret_cast<uintptr_t>(workspace) & 255)) return OZ_ENOMEM;
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  int32_t* rowexp = reinterpret_cast<int32_t*>(ws + L.off_rowexp);
  int32_t* colexp = reinterpret_cast<int32_t*>(ws + L.off_colexp);
  uint16_t* Ap = reinterpret_cast<uint16_t*>(ws + L.off_A);
  uint16_t* Bp = reinterpret_cast<uint16_t*>(ws + L.off_B);
  uint8_t* Cr = ws + L.off_C;
  if (scaling == OZ_SCALE_UNIFORM) {
    if ((rc = ozaki2_scale_split(m, n, k, A, lda, B, ldb, num_moduli, rowexp, colexp, Ap, Bp, stream))) return rc;
  } else {
    if ((rc = ozaki2_exponents_ex(m, n, k, A, lda, B, ldb, num_moduli, scaling, rowexp, colexp, Cr,
                                  total - L.off_C, stream)))
      return rc;
    if ((rc = ozaki2_split_ex(m, n, k, A, lda, B, ldb, num_moduli, scaling, rowexp, colexp, Ap, Bp, stream)))
      return rc;
  }
  if ((rc = ozaki2_residue_gemm(m, n, k, num_moduli, Ap, Bp, Cr, stream))) return rc;
  return ozaki2_crt_ex(m, n, k, num_moduli, scaling, Cr, rowexp, colexp, C, ldc, stream);
}

int ozaki2_dgemm_ex(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc,
                    int num_moduli, int scaling, cudaStream_t stream) {
  int rc = check_dims(m, n, k, lda, ldb, ldc);
  if (rc) return rc;
  if (num_moduli < OZ_MIN_MODULI || num_moduli > OZ_MAX_MODULI || !valid_scaling(scaling)) return OZ_EINVAL;
  if (m == 0 || n == 0) return OZ_OK;
  if (k == 0) return C ? cuda_rc(launch_fill_zero(m, n, C, ldc, stream)) : OZ_EINVAL;
  if (!A || !B || !C) return OZ_EINVAL;  // argument errors before any allocation
  {
    int kA;
    if ((rc = ozaki2_scaling_k(num_moduli, k, scaling, &kA))) return rc;
  }
  const size_t bytes = ozaki2_workspace_bytes_ex(m, n, k, num_moduli, scaling);
  keep_default_pool_cached();
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) {
    cudaGetLastError();
    return OZ_ENOMEM;
  }
  rc = ozaki2_dgemm_ex_ws(m, n, k, A, lda, B, ldb, C, ldc, num_moduli, scaling, ws, bytes, stream);
  const cudaError_t e = cudaFreeAsync(ws, stream);
  if (rc == OZ_OK && e != cudaSuccess) rc = OZ_ECUDA;
  return rc;
}

int ozaki2_dgemm(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc,
                 int num_moduli, cudaStream_t stream) {
  int rc = check_dims(m, n, k, lda, ldb, ldc);
  if (rc) return rc;
  if (num_moduli < OZ_MIN_MODULI || num_moduli > OZ_MAX_MODULI) return OZ_EINVAL;
  if (m == 0 || n == 0) return OZ_OK;
  if (k == 0) return C ? cuda_rc(launch_fill_zero(m, n, C, ldc, stream)) : OZ_EINVAL;
  if (!A || !B || !C) return OZ_EINVAL;  // argument errors before any allocation
  {
    int kA;
    if ((rc = ozaki2_choose_k(num_moduli, k, &kA))) return rc;
  }
  const size_t bytes = ozaki2_workspace_bytes(m, n, k, num_moduli);
  keep_default_pool_cached();
  void* ws = nullptr;
  if (cudaMallocAsync(&ws, bytes, stream) != cudaSuccess) {
    cudaGetLastError();
    return OZ_ENOMEM;
  }
  rc = ozaki2_dgemm_ws(m, n, k, A, lda, B, ldb, C, ldc, num_moduli, ws, bytes, stream);
  const cudaError_t e = cudaFreeAsync(ws, stream);
  if (rc == OZ_OK && e != cudaSuccess) rc = OZ_ECUDA;
  return rc;
}

int ozaki2_dgemm_host(int m, int n, int k, const double* A, int lda, const double* B, int ldb, double* C, int ldc,
                      int num_moduli) {
  int rc = check_dims(m, n, k, lda, ldb, ldc);
  if (rc) return rc;
  if (num_moduli < OZ_MIN_MODULI || num_moduli > OZ_MAX_MODULI) return OZ_EINVAL;
  if (m == 0 || n == 0) return OZ_OK;
  if (!C || (k > 0 && (!A || !B))) return OZ_EINVAL;
  if (k == 0) {  // C = +0 (BLAS with beta = 0); host memory
    for (int j = 0; j < n; ++j) std::memset(C + static_cast<size_t>(j) * ldc, 0, sizeof(double) * m);
    return OZ_OK;
  }
  {
    int kA;
    if ((rc = ozaki2_choose_k(num_moduli, k, &kA))) return rc;
  }
  // Two-dimensional block pipeline: row blocks of A x column blocks of B.  Copies in on one
  // stream (A_0, B_0, A_1, B_1, ...), the path on a second, copies out on a third; the blocks
  // (i, j) are computed in the order their operands arrive (a square wavefront), so only the
  // first two operand blocks and the last block's copy out are not hidden behind compute.
  const int s = num_moduli;
  auto block_count = [](int d) { return d >= 12288 ? 4 : (d >= 2048 ? 2 : 1); };
  const Blocks mb = make_blocks(m, block_count(m));
  const Blocks nbk = make_blocks(n, block_count(n));
  const int kp = static_cast<int>(roundup(k, kPadK));
  size_t off = 0;
  const size_t off_dA = off;
  off = align256(off + sizeof(double) * static_cast<size_t>(m) * k);
  const size_t off_dB = off;
  off = align256(off + sizeof(double) * static_cast<size_t>(k) * n);
  const size_t off_dC = off;
  off = align256(off + sizeof(double) * static_cast<size_t>(m) * n);
  const size_t off_rowexp = off;
  off = align256(off + sizeof(int32_t) * m);
  const size_t off_colexp = off;
  off = align256(off + sizeof(int32_t) * n);
  size_t off_Ap[Blocks::kMax], off_Bp[Blocks::kMax];
  int max_mp = 0, max_np = 0;
  for (int i = 0; i < mb.count; ++i) {
    const int mpi = static_cast<int>(roundup(mb.size[i], kPadM));
    max_mp = mpi > max_mp ? mpi : max_mp;
    off_Ap[i] = off;
    off = align256(off + sizeof(uint16_t) * static_cast<size_t>(s) * mpi * kp);
  }
  for (int j = 0; j < nbk.count; ++j) {
    const int npj = static_cast<int>(roundup(nbk.size[j], kPadN));
    max_np = npj > max_np ? npj : max_np;
    off_Bp[j] = off;
    off = align256(off + sizeof(uint16_t) * static_cast<size_t>(s) * npj * kp);
  }
  const size_t off_Cr = off;
  off = align256(off + static_cast<size_t>(s) * max_mp * max_np);
  const size_t total = off;

  cudaStream_t sin = nullptr, scomp = nullptr, sout = nullptr;
  if (cudaStreamCreateWithFlags(&sin, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&scomp, cudaStreamNonBlocking) != cudaSuccess ||
      cudaStreamCreateWithFlags(&sout, cudaStreamNonBlocking) != cudaSuccess) {
    if (sin) cudaStreamDestroy(sin);
    if (scomp) cudaStreamDestroy(scomp);
    cudaGetLastError();
    return OZ_ECUDA;
  }
  keep_default_pool_cached();
  cudaEvent_t ev[2 * Blocks::kMax + Blocks::kMax * Blocks::kMax] = {};
  const int nev = mb.count + nbk.count + mb.count * nbk.count;
  for (int e = 0; e < nev && !rc; ++e)
    if (cudaEventCreateWithFlags(&ev[e], cudaEventDisableTiming) != cudaSuccess) rc = OZ_ECUDA;
  cudaEvent_t* evA = ev;
  cudaEvent_t* evB = ev + mb.count;
  cudaEvent_t* evC = ev + mb.count + nbk.count;

  uint8_t* ws = nullptr;
  if (!rc && cudaMallocAsync(reinterpret_cast<void**>(&ws), total, scomp) != cudaSuccess) rc = OZ_ENOMEM;
  cudaEvent_t ready = nullptr;  // the allocation is ordered on scomp: the copy streams wait for it
  if (!rc && (cudaEventCreateWithFlags(&ready, cudaEventDisableTiming) != cudaSuccess ||
              cudaEventRecord(ready, scomp) != cudaSuccess || cudaStreamWaitEvent(sin, ready, 0) != cudaSuccess))
    rc = OZ_ECUDA;
  double* dA = reinterpret_cast<double*>(ws + off_dA);
  double* dB = reinterpret_cast<double*>(ws + off_dB);
  double* dC = reinterpret_cast<double*>(ws + off_dC);
  int32_t* rowexp = reinterpret_cast<int32_t*>(ws + off_rowexp);
  int32_t* colexp = reinterpret_cast<int32_t*>(ws + off_colexp);
  uint8_t* Cr = ws + off_Cr;

  // copies in, interleaved: A_0, B_0, A_1, B_1, ... (the order the wavefront consumes them)
  auto copy_A = [&](int i) {
    if (!rc && (cudaMemcpy2DAsync(dA + mb.start[i], sizeof(double) * m, A + mb.start[i], sizeof(double) * lda,
                                  sizeof(double) * mb.size[i], k, cudaMemcpyHostToDevice, sin) != cudaSuccess ||
                cudaEventRecord(evA[i], sin) != cudaSuccess))
      rc = OZ_ECUDA;
  };
  auto copy_B = [&](int j) {
    if (!rc && (cudaMemcpy2DAsync(dB + static_cast<size_t>(nbk.start[j]) * k, sizeof(double) * k,
                                  B + static_cast<size_t>(nbk.start[j]) * ldb, sizeof(double) * ldb,
                                  sizeof(double) * k, nbk.size[j], cudaMemcpyHostToDevice, sin) != cudaSuccess ||
                cudaEventRecord(evB[j], sin) != cudaSuccess))
      rc = OZ_ECUDA;
  };
  for (int q = 0; q < mb.count || q < nbk.count; ++q) {
    if (q < mb.count) copy_A(q);
    if (q < nbk.count) copy_B(q);
  }

  // block order: by the copy after which both operands are in (A_i is copy 2i, B_j copy
  // 2j + 1 while both lists last), then row, then column
  int order[Blocks::kMax * Blocks::kMax];
  int nblocks = 0;
  auto arrival = [&](int i, int j) {
    const int ai = i < nbk.count ? 2 * i : nbk.count + i;
    const int bj = j < mb.count ? 2 * j + 1 : mb.count + j;
    return ai > bj ? ai : bj;
  };
  for (int i = 0; i < mb.count; ++i)
    for (int j = 0; j < nbk.count; ++j) order[nblocks++] = i * nbk.count + j;
  for (int a = 1; a < nblocks; ++a)  // insertion sort, stable: (arrival, i, j)
    for (int b = a; b > 0 && arrival(order[b] / nbk.count, order[b] % nbk.count) <
                                  arrival(order[b - 1] / nbk.count, order[b - 1] % nbk.count);
         --b) {
      const int t = order[b];
      order[b] = order[b - 1];
      order[b - 1] = t;
    }

  // the path, block by block; each operand block is scaled and split when first needed
  bool splitA[Blocks::kMax] = {}, splitB[Blocks::kMax] = {};
  for (int b = 0; b < nblocks && !rc; ++b) {
    const int i = order[b] / nbk.count, j = order[b] % nbk.count;
    const int i0 = mb.start[i], mi = mb.size[i];
    const int j0 = nbk.start[j], nj = nbk.size[j];
    uint16_t* Ap = reinterpret_cast<uint16_t*>(ws + off_Ap[i]);
    uint16_t* Bp = reinterpret_cast<uint16_t*>(ws + off_Bp[j]);
    const double* dBj = dB + static_cast<size_t>(j0) * k;
    if (!splitA[i]) {
      if (cudaStreamWaitEvent(scomp, evA[i], 0) != cudaSuccess) rc = OZ_ECUDA;
      if (!rc) rc = ozaki2_exponents(mi, 0, k, dA + i0, m, nullptr, 1, rowexp + i0, nullptr, scomp);
      if (!rc) rc = ozaki2_split(mi, 0, k, dA + i0, m, nullptr, 1, s, rowexp + i0, nullptr, Ap, nullptr, scomp);
      splitA[i] = true;
    }
    if (!splitB[j]) {
      if (!rc && cudaStreamWaitEvent(scomp, evB[j], 0) != cudaSuccess) rc = OZ_ECUDA;
      if (!rc) rc = ozaki2_scale_split(0, nj, k, nullptr, 1, dBj, k, s, nullptr, colexp + j0, nullptr, Bp, scomp);
      splitB[j] = true;
    }
    if (!rc) rc = ozaki2_residue_gemm(mi, nj, k, s, Ap, Bp, Cr, scomp);
    double* dCij = dC + i0 + static_cast<size_t>(j0) * m;
    if (!rc) rc = ozaki2_crt(mi, nj, k, s, Cr, rowexp + i0, colexp + j0, dCij, m, scomp);
    cudaEvent_t e = evC[i * nbk.count + j];
    if (!rc && (cudaEventRecord(e, scomp) != cudaSuccess || cudaStreamWaitEvent(sout, e, 0) != cudaSuccess ||
                cudaMemcpy2DAsync(C + i0 + static_cast<size_t>(j0) * ldc, sizeof(double) * ldc, dCij,
                                  sizeof(double) * m, sizeof(double) * mi, nj, cudaMemcpyDeviceToHost,
                                  sout) != cudaSuccess))
      rc = OZ_ECUDA;
  }
  (void)kp;
  // release the workspace after the copies out, then wait for everything
  cudaEvent_t done = nullptr;
  if (ws) {
    const bool ordered = cudaEventCreateWithFlags(&done, cudaEventDisableTiming) == cudaSuccess &&
                         cudaEventRecord(done, sout) == cudaSuccess && cudaStreamWaitEvent(scomp, done, 0) == cudaSuccess;
    if (!ordered) cudaStreamSynchronize(sout);  // the copies out read the workspace: finish them first
    cudaFreeAsync(ws, scomp);
  }
  if (cudaStreamSynchronize(sin) != cudaSuccess && !rc) rc = OZ_ECUDA;
  if (cudaStreamSynchronize(sout) != cudaSuccess && !rc) rc = OZ_ECUDA;
  if (cudaStreamSynchronize(scomp) != cudaSuccess && !rc) rc = OZ_ECUDA;
  for (int e = 0; e < nev; ++e)
    if (ev[e]) cudaEventDestroy(ev[e]);
  if (ready) cudaEventDestroy(ready);
  if (done) cudaEventDestroy(done);
  cudaStreamDestroy(sin);
  cudaStreamDestroy(scomp);
  cudaStreamDestroy(sout);
  cudaGetLastError();
  return rc;
}

int ozaki_get_device_status(cudaStream_t stream) {
  if (cudaStreamSynchronize(stream) != cudaSuccess) return OZ_ECUDA;
  int* p = device_status_ptr();
  if (!p) return OZ_ECUDA;
  int v = 0;
  if (cudaMemcpyAsync(&v, p, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaMemsetAsync(p, 0, sizeof(int), stream) != cudaSuccess || cudaStreamSynchronize(stream) != cudaSuccess)
    return OZ_ECUDA;
  return v;
}

const char* ozaki_status_string(int status) {
  switch (status) {
    case OZ_OK: return "OZ_OK";
    case OZ_EINVAL: return "OZ_EINVAL: invalid argument";
    case OZ_ERANGE: return "OZ_ERANGE: too few moduli for this inner dimension";
    case OZ_ECUDA: return "OZ_ECUDA: CUDA runtime error";
    case OZ_ENOMEM: return "OZ_ENOMEM: workspace allocation failed or too small";
    case OZ_ETIMEOUT: return "OZ_ETIMEOUT: a bounded device wait expired";
    case OZ_ENODEV: return "OZ_ENODEV: no usable device";
    default: return "unknown ozaki status";
  }
}

}  // extern "C"
