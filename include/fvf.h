/*
 * fvf.h -- C ABI of libfvf.so, the GB300 (sm_103a) library of per-cell field
 * sweeps: the explicit 2D 5-point and 3D 7-point diffusion steps with
 * ping-pong buffers, the
 * multi-variable WENO input pack and the finite-volume flux-difference source
 * (assigned or accumulated; FP64 and FP32), the directional flux copy back to the physical
 * frame, the conservative-variable copy (alone or fused with the pack) and
 * the SSPRK3 stage update (alone or fused with the flux difference).
 *
 * Sources of the operations (pages, by title and section):
 *   [Q] Qiita, "Fortran 2018でGPUを高速化する Part 3" ("Fortran 2018 GPU
 *       acceleration, part 3"): section 3 (update formula, alpha = 0.1,
 *       stability alpha <= 1/4), section 4 (column-major layout), section 5.1
 *       (edges written 0 each step), section 5.4 (ping-pong), section 6.1
 *       (alpha = 0.1_real32 in FP32).
 *   [M] MFlowCode/MFC pull request #2087, "Collapse only spatial loops in
 *       per-variable GPU kernels": "Changes" (s_pack_weno_input_arr,
 *       s_compute_advection_source_term, s_finalize_riemann_solver,
 *       s_compute_rhs) and "Why
 *       this is faster" (one thread per spatial cell, variables looped inside
 *       the thread).
 *   [D] Mallard documentation, "Design: single-GPU performance and parallel
 *       scaling": "Hardware and method" (a time step is three SSPRK3 stages)
 *       and "Baseline (main)" (per stage, the rhs and axpby kernels).  The
 *       stage coefficients are Shu and Osher's (J. Comput. Phys. 77, 1988).
 *
 * Conventions common to every entry point
 *   - All array pointers are DEVICE pointers owned by the caller (for
 *     instance torch CUDA tensors) on the current CUDA device; the library
 *     allocates no device memory and keeps no pointer after returning.
 *     Pointers to host memory are rejected (FVF_ERR_NOT_DEVICE).
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default
 *     stream).  Calls only enqueue work on it and return; nothing is
 *     synchronised.  A device fault surfaces at the caller's next
 *     synchronisation, as for any CUDA launch.
 *   - Every argument is validated on the host before anything is launched.
 *     On any nonzero status nothing has been enqueued (except FVF_ERR_CUDA,
 *     which reports a failed launch).  fvf_status_string() names a status.
 *   - A 3D field with interior extents (n1, n2, n3) and ghost width g is
 *     stored with extents N_a = n_a + 2g on every axis with n_a > 1 and
 *     N_a = 1 on an axis with n_a == 1 (so a 2D problem passes n3 = 1).
 *     Element (j,k,l) of the stored box is at j + N1*(k + N2*l): j is
 *     contiguous, as in the Fortran arrays of [M].
 *   - Floating-point results are bit-identical to the plain CPU evaluation
 *     of the same formulas in the stated operation order with every
 *     operation rounded to nearest even (no contraction of a multiply and an
 *     add), except that NaN payloads are not preserved by arithmetic.
 */
#ifndef FVF_H_
#define FVF_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Status codes returned by every entry point. */
#define FVF_OK               0  /* success (work enqueued, or nothing to do)      */
#define FVF_ERR_NULL         1  /* a required pointer is NULL                     */
#define FVF_ERR_SIZE         2  /* a size is negative, or a product overflows     */
#define FVF_ERR_DTYPE        3  /* dtype is neither FVF_FP32 nor FVF_FP64         */
#define FVF_ERR_DIR          4  /* dir is not 0, 1 or 2                           */
#define FVF_ERR_NV           5  /* nv outside 0..FVF_MAX_NV                       */
#define FVF_ERR_ALIAS        6  /* an output overlaps an input or the other buffer */
#define FVF_ERR_ALPHA        7  /* alpha or a stage coefficient is not finite     */
#define FVF_ERR_ALIGN        8  /* a pointer is not aligned to its element size   */
#define FVF_ERR_NOT_DEVICE   9  /* a pointer is not device memory of this device  */
#define FVF_ERR_RANGE       10  /* an array runs past the end of its allocation   */
#define FVF_ERR_CUDA        11  /* a CUDA call failed (see fvf_last_cuda_error)   */

/* dtype values of diffuse2d_step. */
#define FVF_FP32 0
#define FVF_FP64 1

/* Largest number of variables the multi-variable calls accept. */
#define FVF_MAX_NV 64

/*
 * diffuse2d_step -- nsteps explicit 5-point diffusion steps with ping-pong
 * buffers ([Q] sections 3, 5.1, 5.4).
 *
 *   u, v    two nx*ny arrays of float (dtype FVF_FP32) or double (FVF_FP64),
 *           column-major: cell (i,j), 0 <= i < nx, 0 <= j < ny, at i + nx*j.
 *           u holds the initial field.  They must not overlap.
 *   alpha   diffusion number; for FP32 it is rounded once to float.  Any
 *           finite value is accepted (stability, alpha <= 1/4, is the
 *           caller's business).
 *   nsteps  number of steps, >= 0.  Step s (1-based) reads u and writes v
 *           when s is odd, reads v and writes u when s is even.  Each step
 *           computes, for 1 <= i <= nx-2 and 1 <= j <= ny-2,
 *               dst(i,j) = c + alpha*((((W + E) + S) + N) - 4c)
 *           with c = src(i,j), W = src(i-1,j), E = src(i+1,j),
 *           S = src(i,j-1), N = src(i,j+1), and writes 0 to every edge cell
 *           of dst.  Edge cells of src are read as they are.
 *   Result: in v after an odd nsteps, in u after an even nsteps (u untouched
 *           for nsteps = 0).  The other buffer holds the previous step.
 *   Empty grids (nx or ny = 0) and nsteps = 0 return FVF_OK and enqueue
 *   nothing.
 *   Pointers must be aligned to the element size.
 */
int diffuse2d_step(void *u, void *v, int64_t nx, int64_t ny, double alpha,
                   int64_t nsteps, int dtype, void *stream);

/*
 * diffuse3d_step -- nsteps explicit 7-point diffusion steps on a 3D grid with
 * ping-pong buffers: the 3D variant of [Q] sections 3, 5.1 and 5.4.
 *
 *   u, v    two nx*ny*nz arrays of float (FVF_FP32) or double (FVF_FP64),
 *           column-major: cell (i,j,k) at i + nx*(j + ny*k).  u holds the
 *           initial field; they must not overlap.
 *   alpha   diffusion number (FP32: rounded once to float); any finite
 *           value (stability needs alpha <= 1/6).
 *   nsteps  >= 0; step s reads u and writes v when s is odd, the reverse when
 *           s is even.  Each step computes, for every interior cell
 *           (1 <= i <= nx-2, 1 <= j <= ny-2, 1 <= k <= nz-2),
 *               dst = c + alpha*((((((W + E) + S) + N) + B) + T) - 6c)
 *           with W/E = src(i-+1,j,k), S/N = src(i,j-+1,k),
 *           B/T = src(i,j,k-+1), 6c rounded on its own, and writes 0 to
 *           every cell of the six boundary faces of dst.
 *   Result: in v after an odd nsteps, in u after an even one.  Empty grids
 *   and nsteps = 0 are no-ops.  Pointers must be aligned to the element size.
 */
int diffuse3d_step(void *u, void *v, int64_t nx, int64_t ny, int64_t nz, double alpha,
                   int64_t nsteps, int dtype, void *stream);

/*
 * weno_pack -- the multi-variable WENO input pack of [M] ("Changes",
 * s_pack_weno_input_arr): out(a,b,c,i) = field_i(...) with the swept axis
 * first.  FP64 bit copy (NaN payloads and signed zeros preserved).
 *
 *   fields   HOST array of nv device pointers; field i is a stored box
 *            (N1 x N2 x N3 doubles, layout above).  Fields may alias each
 *            other; none may overlap out.
 *   nv       number of variables, 0..FVF_MAX_NV (0: nothing to do).
 *   extents  HOST array {n1, n2, n3} of interior extents, each >= 0 (any
 *            zero: nothing to do).
 *   ghost    ghost width g >= 0 on every axis whose interior extent is > 1.
 *   dir      swept axis: 0 = x (j), 1 = y (k), 2 = z (l).
 *   out      M1*M2*M3*nv doubles, out(a,b,c,i) at a + M1*(b + M2*(c + M3*i)):
 *              dir 0: out(a,b,c,i) = field_i(a,    b+g2, c+g3), (M1,M2,M3) = (N1,n2,n3)
 *              dir 1: out(a,b,c,i) = field_i(b+g1, a,    c+g3), (M1,M2,M3) = (N2,n1,n3)
 *              dir 2: out(a,b,c,i) = field_i(c+g1, b+g2, a   ), (M1,M2,M3) = (N3,n2,n1)
 *            with g_a = g where n_a > 1, else 0: the swept axis covers its
 *            ghost cells, the transverse axes their interior cells.
 */
int weno_pack(const double *const *fields, int nv, const int64_t extents[3], int ghost,
              int dir, double *out, void *stream);

/*
 * weno_pack_f32 -- weno_pack on FP32 fields: the same element mapping, a
 * 4-byte bit copy.  Arguments as for weno_pack with float in place of
 * double (pointers 4-byte aligned).  [Q] section 6 measures FP32 against
 * FP64 for the same sweeps.
 */
int weno_pack_f32(const float *const *fields, int nv, const int64_t extents[3], int ghost,
                  int dir, float *out, void *stream);

/*
 * advect_rhs -- the finite-volume flux-difference source of [M]
 * ("Changes", s_compute_advection_source_term), one direction per call,
 * assigned (not accumulated):
 *     dir 0: rhs(j,k,l,i) = inv_d(j) * (F(j-1,k,l,i) - F(j,k,l,i))
 *     dir 1: rhs(j,k,l,i) = inv_d(k) * (F(j,k-1,l,i) - F(j,k,l,i))
 *     dir 2: rhs(j,k,l,i) = inv_d(l) * (F(j,k,l-1,i) - F(j,k,l,i))
 * one subtraction then one multiplication, for 0 <= j < n1, 0 <= k < n2,
 * 0 <= l < n3, 0 <= i < nv.
 *
 *   flux     face fluxes, contiguous doubles with the variable slowest and
 *            one extra entry along the swept axis: extents (n1+1, n2, n3),
 *            (n1, n2+1, n3) or (n1, n2, n3+1) per variable; face f
 *            (-1 <= f <= n-1) is stored at position f+1 on that axis.
 *   inv_d    inverse cell widths along the swept axis (n_dir doubles).
 *   nv       0..FVF_MAX_NV (0: nothing to do).
 *   extents  HOST array {n1, n2, n3} of cell counts, each >= 0.
 *   dir      0, 1 or 2.
 *   rhs      n1*n2*n3*nv doubles, rhs(j,k,l,i) at j + n1*(k + n2*(l + n3*i));
 *            must not overlap flux or inv_d.
 */
int advect_rhs(const double *flux, const double *inv_d, int nv, const int64_t extents[3],
               int dir, double *rhs, void *stream);

/*
 * advect_rhs_add -- the accumulating form of advect_rhs: the same term,
 * added once to the existing rhs,
 *     rhs(j,k,l,i) = rhs(j,k,l,i) + inv_d(c) * (F(c-1) - F(c)),
 * so that the x, y and z calls build the finite-volume right-hand side (the
 * x/y/z flux differences of [M] "Changes", s_compute_advection_source_term,
 * are the terms of one sum).  Arguments, layouts and validation as for
 * advect_rhs; rhs is read and written.
 */
int advect_rhs_add(const double *flux, const double *inv_d, int nv, const int64_t extents[3],
                   int dir, double *rhs, void *stream);

/*
 * advect_rhs_f32, advect_rhs_add_f32 -- advect_rhs and advect_rhs_add in
 * binary32: flux, inv_d and rhs are float arrays of the same layouts, and the
 * subtraction, multiplication (and, for the accumulating form, addition) are
 * binary32 operations, each rounded to nearest even.
 */
int advect_rhs_f32(const float *flux, const float *inv_d, int nv, const int64_t extents[3],
                   int dir, float *rhs, void *stream);
int advect_rhs_add_f32(const float *flux, const float *inv_d, int nv, const int64_t extents[3],
                       int dir, float *rhs, void *stream);

/*
 * flux_unpack -- the directional flux copy from the sweep frame back to the
 * physical frame ([M] "Changes", s_finalize_riemann_solver): the inverse of
 * the pack's axis exchange, for face arrays.  A bit copy.
 *
 *   sweep_flux  contiguous doubles, swept axis first with its n+1 faces,
 *               variable slowest:
 *                 dir 0: in(f,k,l,i), extents (n1+1, n2, n3)
 *                 dir 1: in(f,j,l,i), extents (n2+1, n1, n3)
 *                 dir 2: in(f,k,j,i), extents (n3+1, n2, n1)
 *   nv          0..FVF_MAX_NV (0: nothing to do).
 *   extents     HOST array {n1, n2, n3} of cell counts, each >= 0.
 *   out         the face array in the physical frame (the layout advect_rhs
 *               reads): extents (n1+1,n2,n3), (n1,n2+1,n3) or (n1,n2,n3+1),
 *               j fastest, variable slowest; must not overlap sweep_flux.
 */
int flux_unpack(const double *sweep_flux, int nv, const int64_t extents[3], int dir,
                double *out, void *stream);

/*
 * fields_copy -- the conservative-variable copy of [M] ("Changes",
 * s_compute_rhs): copy_i = field_i element by element over the whole stored
 * box, ghost cells included, for every variable.  A bit copy (NaN payloads and
 * signed zeros preserved).
 *
 *   fields   HOST array of nv device pointers, each a stored box of
 *            N1*N2*N3 doubles (layout above).  Fields may alias each other.
 *   nv       0..FVF_MAX_NV (0: nothing to do).
 *   extents  HOST array {n1, n2, n3} of interior extents, each >= 0.
 *   ghost    ghost width g >= 0 (it only sets the stored extents N_a).
 *   copies   HOST array of nv device pointers, each N1*N2*N3 doubles.  A
 *            copy must not overlap any field or any other copy.
 */
int fields_copy(const double *const *fields, int nv, const int64_t extents[3], int ghost,
                double *const *copies, void *stream);

/*
 * weno_pack_copy -- weno_pack and fields_copy of the same fields in one pass:
 * each stored element is read once, written to its copy and, when it lies in
 * the pack's region, to out.  The results equal those of weno_pack(fields,
 * nv, extents, ghost, dir, out) and fields_copy(fields, nv, extents, ghost,
 * copies).  [M] ("Changes") lists both loops, in s_compute_rhs and
 * s_pack_weno_input_arr, over the same conservative-variable fields.
 *
 *   Arguments as for weno_pack, plus copies as for fields_copy.  out must
 *   not overlap a field or a copy.
 */
int weno_pack_copy(const double *const *fields, int nv, const int64_t extents[3], int ghost,
                   int dir, double *out, double *const *copies, void *stream);

/*
 * ssprk3_axpby -- one SSPRK3 stage update ([D], axpby per stage):
 *     out(c,i) = a*u0(c,i) + b*(u(c,i) + dt*rhs(c,i))
 * evaluated as t = u + dt*rhs, then a*u0 and b*t, then their sum, each
 * operation rounded to nearest even.  The three stages of a step use
 * (a, b) = (0, 1), (3/4, 1/4), (1/3, 2/3) with u0 = u^n and u the previous
 * stage (u^n itself in stage 1); 1/3 and 2/3 are the doubles nearest them.
 * The formula is applied as written for any finite a, b, dt (0*u0 is still
 * computed when a = 0).
 *
 *   u0, u, rhs, out  n1*n2*n3*nv doubles each, cell (j,k,l) of variable i at
 *                    j + n1*(k + n2*(l + n3*i)) (the rhs layout of
 *                    advect_rhs).  u0 and u may be the same array.  out may
 *                    be u or u0 itself (same start address: an in-place
 *                    stage) but must not overlap them otherwise, nor rhs.
 *   nv               0..FVF_MAX_NV (0: nothing to do).
 *   extents          HOST array {n1, n2, n3} of cell counts, each >= 0.
 *   a, b, dt         finite (else FVF_ERR_ALPHA).
 */
int ssprk3_axpby(const double *u0, const double *u, const double *rhs, int nv,
                 const int64_t extents[3], double a, double b, double dt, double *out,
                 void *stream);

/*
 * ssprk3_stage -- the stage update fused with the flux difference: rhs is
 * formed in registers from the face fluxes, exactly as advect_rhs for x
 * followed by advect_rhs_add for y and then z would form it,
 *     rhs = inv_x(j)*(Fx(j-1) - Fx(j))
 *           [+ inv_y(k)*(Fy(k-1) - Fy(k))] [+ inv_z(l)*(Fz(l-1) - Fz(l))],
 * then out = a*u0 + b*(u + dt*rhs) as in ssprk3_axpby.  No rhs array is
 * read or written.
 *
 *   flux    HOST array of 3 device pointers: the x, y and z face fluxes in
 *           the layouts of advect_rhs.  flux[0] is required; flux[1] or
 *           flux[2] NULL leaves that direction out (a 2D or 1D problem).
 *   inv_d   HOST array of 3 device pointers: inverse cell widths along x
 *           (n1 doubles), y (n2) and z (n3); needed where the flux is given.
 *   Other arguments as for ssprk3_axpby; out must not overlap a flux or an
 *   inverse-width array.
 */
int ssprk3_stage(const double *u0, const double *u, const double *const flux[3],
                 const double *const inv_d[3], int nv, const int64_t extents[3], double a,
                 double b, double dt, double *out, void *stream);

/* Static, NUL-terminated name of a status code ("unknown status" if none). */
const char *fvf_status_string(int status);

/* The cudaError_t value behind the calling thread's last FVF_ERR_CUDA
 * (0 if none). */
int fvf_last_cuda_error(void);

/*
 * fvf_device_error -- reads and clears the device-side error flags of the
 * current device.  *flag gets a bit mask, 0 when nothing was recorded:
 *   1  a kernel that waits on its own asynchronous copies (diffuse3d_step's
 *      bulk-copy kernel) gave up a bounded wait, let its copies in flight
 *      finish (also bounded) and returned without completing its work: the
 *      results of that launch are invalid;
 *   2  (index-checking debug builds only, libfvf_check.so) a kernel met a
 *      global index outside its array and skipped that access;
 *   4  (with 1) one of the waits for the copies still in flight expired as
 *      well: a block may have returned while a copy into its shared memory
 *      was pending.
 * Synchronises the device.  Returns FVF_OK, FVF_ERR_NULL or FVF_ERR_CUDA.
 */
int fvf_device_error(int *flag);

/* Number of kernels this library has launched since it was loaded (all
 * threads).  Lets a caller count the library's launches in a region. */
uint64_t fvf_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FVF_H_ */
