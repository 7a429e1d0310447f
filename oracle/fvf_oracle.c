/*
 * fvf_oracle.c -- plain, slow, obviously correct CPU oracle for the three
 * per-cell field sweeps.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check
 * and the benchmark's CPU-baseline leg call it; the GPU library never links,
 * includes or calls anything here, and nothing here includes the GPU code.
 *
 * Build: gcc -O2 -ffp-contract=off [-fopenmp] -fPIC -shared.  Contraction is
 * switched off so that every `a*b + c` below is a separately rounded multiply
 * and add, as the Fortran reference on the Qiita page performs them.
 *
 * Sources (pages, by title and section):
 *  [Q]  Qiita, "Fortran 2018でGPUを高速化する Part 3 -- GPUカーネルの
 *       メモリアクセスとFP32・FP64を比較する" ("Fortran 2018 GPU acceleration,
 *       part 3"): section 3 (the 5-point update and alpha), section 4
 *       (column-major layout, i contiguous), section 5.1 (all-cells variant,
 *       edges written 0 each step), section 5.4 (ping-pong: odd steps u->v,
 *       even steps v->u), appendix A (CPU reference program: j outer loop,
 *       i inner loop, same update).
 *  [M]  MFlowCode/MFC pull request #2087, "Collapse only spatial loops in
 *       per-variable GPU kernels": "Changes" (the WENO input pack
 *       v_rs_weno(j,k,l,i) = v_vf(i)%sf(j,k,l) and the x/y/z flux
 *       differences in s_compute_advection_source_term, inverse spacing taken
 *       once per cell; s_finalize_riemann_solver, the directional flux copies;
 *       s_compute_rhs, the conservative-variable copy).
 *  [D]  Mallard documentation, "Design: single-GPU performance and parallel
 *       scaling": "Hardware and method" (a step is SSPRK3, three stages) and
 *       "Baseline (main)" (per stage, after the flux sums, the rhs and axpby
 *       kernels).  The stage coefficients are those of the three-stage,
 *       third-order strong-stability-preserving Runge-Kutta scheme of Shu and
 *       Osher (J. Comput. Phys. 77, 1988): u1 = u^n + dt L(u^n),
 *       u2 = 3/4 u^n + 1/4 (u1 + dt L(u1)), u^{n+1} = 1/3 u^n + 2/3 (u2 + dt L(u2)).
 *
 * Conventions (0-based C indices; the pages use 1-based Fortran):
 *  - 2D field u(i,j), 0 <= i < nx, 0 <= j < ny, stored at u[i + nx*j].
 *  - A 3D field with interior extents (n1,n2,n3) and ghost width g is stored
 *    with extents N_a = n_a + 2g on every axis with n_a > 1 and N_a = 1 on an
 *    axis with n_a == 1 (a 2D problem has n3 == 1).  Element (j,k,l) of the
 *    stored box sits at j + N1*(k + N2*l); interior cell (j,k,l) is stored
 *    element (j+g1, k+g2, l+g3) with g_a = g where n_a > 1, else 0.
 */
#include <stddef.h>
#include <stdint.h>

/* ---------------------------------------------------------------------- */
/* 2D explicit diffusion                                                  */
/* ---------------------------------------------------------------------- */

/*
 * One application of the update of [Q] section 3:
 *     dst(i,j) = src(i,j) + alpha*(src(i-1,j) + src(i+1,j)
 *                                  + src(i,j-1) + src(i,j+1) - 4*src(i,j))
 * for interior cells, and dst = 0 on the four edges ([Q] section 5.1 and the
 * appendix-A CPU program).  C evaluates the bracket left to right, exactly as
 * Fortran does: ((((W + E) + S) + N) - 4c), then alpha times that, then c plus
 * the product, each operation rounded to nearest even.
 */
static void step_f64(const double *src, double *dst, int64_t nx, int64_t ny,
                     double alpha, int nthreads)
{
    int64_t j;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (j = 0; j < ny; ++j) {
        for (int64_t i = 0; i < nx; ++i) {
            const int64_t c = i + nx * j;
            if (i == 0 || i == nx - 1 || j == 0 || j == ny - 1) {
                dst[c] = 0.0;
            } else {
                dst[c] = src[c] + alpha * (src[c - 1] + src[c + 1] + src[c - nx]
                                           + src[c + nx] - 4.0 * src[c]);
            }
        }
    }
}

static void step_f32(const float *src, float *dst, int64_t nx, int64_t ny,
                     float alpha, int nthreads)
{
    int64_t j;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (j = 0; j < ny; ++j) {
        for (int64_t i = 0; i < nx; ++i) {
            const int64_t c = i + nx * j;
            if (i == 0 || i == nx - 1 || j == 0 || j == ny - 1) {
                dst[c] = 0.0f;
            } else {
                dst[c] = src[c] + alpha * (src[c - 1] + src[c + 1] + src[c - nx]
                                           + src[c + nx] - 4.0f * src[c]);
            }
        }
    }
}

/*
 * nsteps applications with the ping-pong of [Q] section 5.4: step s
 * (1-based) reads u and writes v when s is odd, reads v and writes u when s
 * is even.  The result is in v after an odd count and in u after an even
 * count.  Returns 1 when the result is in v, 0 when it is in u.
 */
int oracle_diffuse2d_f64(double *u, double *v, int64_t nx, int64_t ny,
                         double alpha, int64_t nsteps, int nthreads)
{
    for (int64_t s = 1; s <= nsteps; ++s) {
        if (s % 2 == 1)
            step_f64(u, v, nx, ny, alpha, nthreads);
        else
            step_f64(v, u, nx, ny, alpha, nthreads);
    }
    return (int)(nsteps % 2);
}

/* FP32 variant; alpha is the FP32 value (0.1_real32 in [Q] section 6.1). */
int oracle_diffuse2d_f32(float *u, float *v, int64_t nx, int64_t ny,
                         float alpha, int64_t nsteps, int nthreads)
{
    for (int64_t s = 1; s <= nsteps; ++s) {
        if (s % 2 == 1)
            step_f32(u, v, nx, ny, alpha, nthreads);
        else
            step_f32(v, u, nx, ny, alpha, nthreads);
    }
    return (int)(nsteps % 2);
}

/* ---------------------------------------------------------------------- */
/* 3D explicit diffusion (7-point)                                        */
/* ---------------------------------------------------------------------- */

/*
 * The 7-point variant of the update of [Q] section 3 on a 3D grid (the
 * 2D scheme with the two z neighbours added and the centre weight 6):
 *     dst(i,j,k) = c + alpha*(W + E + S + N + B + T - 6c)
 * with W/E = src(i-+1,j,k), S/N = src(i,j-+1,k), B/T = src(i,j,k-+1), for
 * interior cells, and dst = 0 on the six boundary faces ([Q] section 5.1
 * extended to 3D).  Evaluated left to right as in the 2D update:
 * (((((W + E) + S) + N) + B) + T) - 6c, then alpha times that, then c plus
 * the product; 6c is its own rounded product (unlike 4c it is not exact).
 * Column-major layout, i fastest: cell (i,j,k) at i + nx*(j + ny*k).
 */
static void step3d_f64(const double *src, double *dst, int64_t nx, int64_t ny, int64_t nz,
                       double alpha, int nthreads)
{
    const int64_t sxy = nx * ny;
    int64_t k;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (k = 0; k < nz; ++k) {
        for (int64_t j = 0; j < ny; ++j) {
            for (int64_t i = 0; i < nx; ++i) {
                const int64_t c = i + nx * (j + ny * k);
                if (i == 0 || i == nx - 1 || j == 0 || j == ny - 1 || k == 0 || k == nz - 1) {
                    dst[c] = 0.0;
                } else {
                    dst[c] = src[c] + alpha * (src[c - 1] + src[c + 1] + src[c - nx]
                                               + src[c + nx] + src[c - sxy] + src[c + sxy]
                                               - 6.0 * src[c]);
                }
            }
        }
    }
}

static void step3d_f32(const float *src, float *dst, int64_t nx, int64_t ny, int64_t nz,
                       float alpha, int nthreads)
{
    const int64_t sxy = nx * ny;
    int64_t k;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nthreads)
#else
    (void)nthreads;
#endif
    for (k = 0; k < nz; ++k) {
        for (int64_t j = 0; j < ny; ++j) {
            for (int64_t i = 0; i < nx; ++i) {
                const int64_t c = i + nx * (j + ny * k);
                if (i == 0 || i == nx - 1 || j == 0 || j == ny - 1 || k == 0 || k == nz - 1) {
                    dst[c] = 0.0f;
                } else {
                    dst[c] = src[c] + alpha * (src[c - 1] + src[c + 1] + src[c - nx]
                                               + src[c + nx] + src[c - sxy] + src[c + sxy]
                                               - 6.0f * src[c]);
                }
            }
        }
    }
}

/* nsteps ping-pong applications ([Q] section 5.4, as oracle_diffuse2d_f64).
 * Returns 1 when the result is in v, 0 when it is in u. */
int oracle_diffuse3d_f64(double *u, double *v, int64_t nx, int64_t ny, int64_t nz,
                         double alpha, int64_t nsteps, int nthreads)
{
    for (int64_t s = 1; s <= nsteps; ++s) {
        if (s % 2 == 1)
            step3d_f64(u, v, nx, ny, nz, alpha, nthreads);
        else
            step3d_f64(v, u, nx, ny, nz, alpha, nthreads);
    }
    return (int)(nsteps % 2);
}

int oracle_diffuse3d_f32(float *u, float *v, int64_t nx, int64_t ny, int64_t nz,
                         float alpha, int64_t nsteps, int nthreads)
{
    for (int64_t s = 1; s <= nsteps; ++s) {
        if (s % 2 == 1)
            step3d_f32(u, v, nx, ny, nz, alpha, nthreads);
        else
            step3d_f32(v, u, nx, ny, nz, alpha, nthreads);
    }
    return (int)(nsteps % 2);
}

/* ---------------------------------------------------------------------- */
/* 3D box helpers                                                         */
/* ---------------------------------------------------------------------- */

static int64_t stored_extent(int64_t n, int64_t g) { return n > 1 ? n + 2 * g : 1; }
static int64_t ghost_offset(int64_t n, int64_t g) { return n > 1 ? g : 0; }

/* ---------------------------------------------------------------------- */
/* WENO input pack                                                        */
/* ---------------------------------------------------------------------- */

/*
 * The pack of [M] "Changes": out(j,k,l,i) = field_i(j,k,l), written as a
 * plain element copy.  The page shows the x direction only; for y and z the
 * first index of the output runs along the swept axis, i.e. the output is
 * the field with the swept axis and the j axis exchanged:
 *   dir 0 (x): out(a, b, c, i) = field_i(a,      b+g2, c+g3), extents (N1, n2, n3)
 *   dir 1 (y): out(a, b, c, i) = field_i(b+g1,   a,    c+g3), extents (N2, n1, n3)
 *   dir 2 (z): out(a, b, c, i) = field_i(c+g1,   b+g2, a   ), extents (N3, n2, n1)
 * where the swept axis covers its ghost cells and the two transverse axes
 * cover the interior only.  out(a,b,c,i) is stored at
 * a + M1*(b + M2*(c + M3*i)) with (M1,M2,M3) the extents above.
 * Returns 0, or -1 for an unknown direction.
 */
int oracle_weno_pack(const double *const *fields, int nv, int64_t n1, int64_t n2,
                     int64_t n3, int64_t g, int dir, double *out)
{
    const int64_t N1 = stored_extent(n1, g), N2 = stored_extent(n2, g);
    const int64_t N3 = stored_extent(n3, g);
    const int64_t g1 = ghost_offset(n1, g), g2 = ghost_offset(n2, g);
    const int64_t g3 = ghost_offset(n3, g);
    int64_t M1, M2, M3;
    if (dir == 0) {
        M1 = N1; M2 = n2; M3 = n3;
    } else if (dir == 1) {
        M1 = N2; M2 = n1; M3 = n3;
    } else if (dir == 2) {
        M1 = N3; M2 = n2; M3 = n1;
    } else {
        return -1;
    }
    for (int i = 0; i < nv; ++i) {
        const double *f = fields[i];
        for (int64_t c = 0; c < M3; ++c) {
            for (int64_t b = 0; b < M2; ++b) {
                for (int64_t a = 0; a < M1; ++a) {
                    int64_t j, k, l;
                    if (dir == 0) {
                        j = a; k = b + g2; l = c + g3;
                    } else if (dir == 1) {
                        j = b + g1; k = a; l = c + g3;
                    } else {
                        j = c + g1; k = b + g2; l = a;
                    }
                    out[a + M1 * (b + M2 * (c + M3 * (int64_t)i))] =
                        f[j + N1 * (k + N2 * l)];
                }
            }
        }
    }
    return 0;
}

/* ---------------------------------------------------------------------- */
/* Flux-difference source                                                 */
/* ---------------------------------------------------------------------- */

/*
 * The x/y/z flux differences of [M] "Changes"
 * (s_compute_advection_source_term):
 *   dir 0: rhs(j,k,l,i) = inv_d(j) * (F(j-1,k,l,i) - F(j,k,l,i))
 *   dir 1: rhs(j,k,l,i) = inv_d(k) * (F(j,k-1,l,i) - F(j,k,l,i))
 *   dir 2: rhs(j,k,l,i) = inv_d(l) * (F(j,k,l-1,i) - F(j,k,l,i))
 * over interior cells 0 <= j < n1, 0 <= k < n2, 0 <= l < n3.  The face array
 * has one more entry than cells along the swept axis: face f (-1 <= f <= n-1)
 * is stored at position f+1 on that axis, and the array is contiguous with
 * the variable index slowest.  rhs(j,k,l,i) is stored at
 * j + n1*(k + n2*(l + n3*i)).  One subtraction, then one multiplication.
 * Returns 0, or -1 for an unknown direction.
 */
int oracle_advect_rhs(const double *flux, const double *inv_d, int nv, int64_t n1,
                      int64_t n2, int64_t n3, int dir, double *rhs)
{
    int64_t F1 = n1, F2 = n2, F3 = n3;
    if (dir == 0)
        F1 = n1 + 1;
    else if (dir == 1)
        F2 = n2 + 1;
    else if (dir == 2)
        F3 = n3 + 1;
    else
        return -1;
    for (int i = 0; i < nv; ++i) {
        for (int64_t l = 0; l < n3; ++l) {
            for (int64_t k = 0; k < n2; ++k) {
                for (int64_t j = 0; j < n1; ++j) {
                    /* stored positions of the low face (f = cell-1) and the
                     * high face (f = cell) of this cell along the swept axis */
                    int64_t jl = j, kl = k, ll = l, jh = j, kh = k, lh = l;
                    double w;
                    if (dir == 0) {
                        jl = j; jh = j + 1; w = inv_d[j];
                    } else if (dir == 1) {
                        kl = k; kh = k + 1; w = inv_d[k];
                    } else {
                        ll = l; lh = l + 1; w = inv_d[l];
                    }
                    const double lo = flux[jl + F1 * (kl + F2 * (ll + F3 * (int64_t)i))];
                    const double hi = flux[jh + F1 * (kh + F2 * (lh + F3 * (int64_t)i))];
                    rhs[j + n1 * (k + n2 * (l + n3 * (int64_t)i))] = w * (lo - hi);
                }
            }
        }
    }
    return 0;
}

/*
 * Accumulating form of the flux difference: rhs(j,k,l,i) = rhs(j,k,l,i) +
 * inv_d(c) * (F(c-1) - F(c)), so that successive directions build the
 * finite-volume right-hand side (the x/y/z flux differences of
 * s_compute_advection_source_term in [M] "Changes" are terms of one sum).
 * The term is formed exactly as in oracle_advect_rhs, then added once.
 */
int oracle_advect_rhs_add(const double *flux, const double *inv_d, int nv, int64_t n1,
                          int64_t n2, int64_t n3, int dir, double *rhs)
{
    int64_t F1 = n1, F2 = n2, F3 = n3;
    if (dir == 0)
        F1 = n1 + 1;
    else if (dir == 1)
        F2 = n2 + 1;
    else if (dir == 2)
        F3 = n3 + 1;
    else
        return -1;
    for (int i = 0; i < nv; ++i) {
        for (int64_t l = 0; l < n3; ++l) {
            for (int64_t k = 0; k < n2; ++k) {
                for (int64_t j = 0; j < n1; ++j) {
                    const int64_t c = dir == 0 ? j : (dir == 1 ? k : l);
                    const int64_t sj = dir == 0 ? 1 : 0, sk = dir == 1 ? 1 : 0, sl = dir == 2 ? 1 : 0;
                    const double lo = flux[j + F1 * (k + F2 * (l + F3 * (int64_t)i))];
                    const double hi = flux[(j + sj) + F1 * ((k + sk) + F2 * ((l + sl) + F3 * (int64_t)i))];
                    const double term = inv_d[c] * (lo - hi);
                    double *r = &rhs[j + n1 * (k + n2 * (l + n3 * (int64_t)i))];
                    *r = *r + term;
                }
            }
        }
    }
    return 0;
}

/*
 * Directional flux copy back to the physical frame (s_finalize_riemann_solver
 * in [M] "Changes"): the inverse of the pack's permutation for face arrays.
 * A sweep-frame face array has the swept axis first, with its n+1 faces:
 *   dir 0: in(f, k, l, i), extents (n1+1, n2, n3)  ->  out(f, k, l, i)   (same layout)
 *   dir 1: in(f, j, l, i), extents (n2+1, n1, n3)  ->  out(j, f, l, i), extents (n1, n2+1, n3)
 *   dir 2: in(f, k, j, i), extents (n3+1, n2, n1)  ->  out(j, k, f, i), extents (n1, n2, n3+1)
 * Arrays are contiguous with the first index fastest and the variable slowest.
 * A plain element copy.  Returns 0, or -1 for an unknown direction.
 */
int oracle_flux_unpack(const double *in, int nv, int64_t n1, int64_t n2, int64_t n3, int dir,
                       double *out)
{
    int64_t F1 = n1, F2 = n2, F3 = n3;   /* physical face-array extents */
    if (dir == 0)
        F1 = n1 + 1;
    else if (dir == 1)
        F2 = n2 + 1;
    else if (dir == 2)
        F3 = n3 + 1;
    else
        return -1;
    for (int i = 0; i < nv; ++i) {
        for (int64_t l = 0; l < F3; ++l) {
            for (int64_t k = 0; k < F2; ++k) {
                for (int64_t j = 0; j < F1; ++j) {
                    int64_t src;
                    if (dir == 0)
                        src = j + F1 * (k + F2 * (l + F3 * (int64_t)i));
                    else if (dir == 1)   /* in(f=k, j, l): extents (F2, F1, F3) */
                        src = k + F2 * (j + F1 * (l + F3 * (int64_t)i));
                    else                 /* in(f=l, k, j): extents (F3, F2, F1) */
                        src = l + F3 * (k + F2 * (j + F1 * (int64_t)i));
                    out[j + F1 * (k + F2 * (l + F3 * (int64_t)i))] = in[src];
                }
            }
        }
    }
    return 0;
}

/*
 * FP32 forms of the pack and of the flux difference ([Q] section 6 compares
 * FP32 with FP64 throughout; the same sweeps on binary32 data).  The pack is
 * the same element mapping as oracle_weno_pack, as a 4-byte copy.  The flux
 * difference forms inv_d(c) * (F(c-1) - F(c)) in binary32 arithmetic (one
 * rounded subtraction, one rounded multiplication) and assigns it, or with
 * accumulate != 0 adds it once to the existing rhs, as oracle_advect_rhs and
 * oracle_advect_rhs_add do in binary64.
 */
int oracle_weno_pack_f32(const float *const *fields, int nv, int64_t n1, int64_t n2,
                         int64_t n3, int64_t g, int dir, float *out)
{
    const int64_t N1 = stored_extent(n1, g), N2 = stored_extent(n2, g);
    const int64_t N3 = stored_extent(n3, g);
    const int64_t g1 = ghost_offset(n1, g), g2 = ghost_offset(n2, g);
    const int64_t g3 = ghost_offset(n3, g);
    int64_t M1, M2, M3;
    (void)N3;
    if (dir == 0) {
        M1 = N1; M2 = n2; M3 = n3;
    } else if (dir == 1) {
        M1 = N2; M2 = n1; M3 = n3;
    } else if (dir == 2) {
        M1 = N3; M2 = n2; M3 = n1;
    } else {
        return -1;
    }
    for (int i = 0; i < nv; ++i) {
        const float *f = fields[i];
        for (int64_t c = 0; c < M3; ++c) {
            for (int64_t b = 0; b < M2; ++b) {
                for (int64_t a = 0; a < M1; ++a) {
                    int64_t j, k, l;
                    if (dir == 0) {
                        j = a; k = b + g2; l = c + g3;
                    } else if (dir == 1) {
                        j = b + g1; k = a; l = c + g3;
                    } else {
                        j = c + g1; k = b + g2; l = a;
                    }
                    out[a + M1 * (b + M2 * (c + M3 * (int64_t)i))] =
                        f[j + N1 * (k + N2 * l)];
                }
            }
        }
    }
    return 0;
}

int oracle_advect_rhs_f32(const float *flux, const float *inv_d, int nv, int64_t n1,
                          int64_t n2, int64_t n3, int dir, int accumulate, float *rhs)
{
    int64_t F1 = n1, F2 = n2, F3 = n3;
    if (dir == 0)
        F1 = n1 + 1;
    else if (dir == 1)
        F2 = n2 + 1;
    else if (dir == 2)
        F3 = n3 + 1;
    else
        return -1;
    for (int i = 0; i < nv; ++i) {
        for (int64_t l = 0; l < n3; ++l) {
            for (int64_t k = 0; k < n2; ++k) {
                for (int64_t j = 0; j < n1; ++j) {
                    const int64_t c = dir == 0 ? j : (dir == 1 ? k : l);
                    const int64_t sj = dir == 0, sk = dir == 1, sl = dir == 2;
                    const float lo = flux[j + F1 * (k + F2 * (l + F3 * (int64_t)i))];
                    const float hi =
                        flux[(j + sj) + F1 * ((k + sk) + F2 * ((l + sl) + F3 * (int64_t)i))];
                    const float term = inv_d[c] * (lo - hi);
                    float *r = &rhs[j + n1 * (k + n2 * (l + n3 * (int64_t)i))];
                    *r = accumulate ? *r + term : term;
                }
            }
        }
    }
    return 0;
}

/*
 * The conservative-variable copy of [M] "Changes" (s_compute_rhs): field i
 * copied element by element, the whole stored box (ghost cells included),
 * into dst_i.  Returns 0.
 */
int oracle_fields_copy(const double *const *src, int nv, int64_t n1, int64_t n2, int64_t n3,
                       int64_t g, double *const *dst)
{
    const int64_t total = stored_extent(n1, g) * stored_extent(n2, g) * stored_extent(n3, g);
    for (int i = 0; i < nv; ++i)
        for (int64_t e = 0; e < total; ++e)
            dst[i][e] = src[i][e];
    return 0;
}

/*
 * One SSPRK3 stage update ([D] "Baseline (main)", axpby per stage) on
 * `count` cell-variable entries:
 *     out = a*u0 + b*(u + dt*rhs)
 * evaluated as t = u + dt*rhs, then a*u0 and b*t, then their sum, every
 * operation rounded separately.  (a, b) is (0, 1), (3/4, 1/4) or (1/3, 2/3)
 * for the three stages, with u0 = u^n and u the previous stage.  out may be
 * u or u0 itself: each entry is read before it is written.  Returns 0.
 */
int oracle_rk_axpby(const double *u0, const double *u, const double *rhs, int64_t count,
                    double a, double b, double dt, double *out)
{
    for (int64_t e = 0; e < count; ++e) {
        const double t = u[e] + dt * rhs[e];
        const double p = a * u0[e];
        const double q = b * t;
        out[e] = p + q;
    }
    return 0;
}

/* Number of OpenMP threads the diffusion loops may use (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
