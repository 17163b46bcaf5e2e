/*
 * Seeded synthetic attention inputs shaped like video-DiT token grids.
 *
 * This file only draws random vectors. It holds no step of the attention method
 * and is shared, unchanged, by the CPU oracle's tests and the CUDA path's tests
 * and benchmark: both sides read the same bf16 bytes.
 *
 * Definition (counter-based, so any token range can be produced independently):
 *   draw64(seed, stream, i) = SM(SM(SM(seed) ^ stream) ^ i), where SM is the
 *       SplitMix64 finaliser of Steele, Lea and Flood, "Fast splittable
 *       pseudorandom number generators" (OOPSLA 2014).
 *   A pair of standard normals comes from one draw by the Box-Muller transform:
 *       u1 = (hi32 + 1) / 2^32 in (0, 1], u2 = lo32 / 2^32,
 *       z0 = sqrt(-2 ln u1) cos(2 pi u2), z1 = sqrt(-2 ln u1) sin(2 pi u2).
 *   Element t (t even: z0, t odd: z1) of a row with counter r uses draw index
 *       (r * d + t) / 2.
 *   Streams: stream(tensor, b, h) = tensor * 2^48 + b * 2^24 + h.
 *       tensor 0: per-cell centre vectors c, row counter = cell id;
 *       tensor 1, 2, 3: the noise of Q, K, V, row counter = token index.
 *   Token s sits at (t, y, x) of a T x Hg x W grid in raster order
 *       (s = (t * Hg + y) * W + x); its cell is (t / ct, y / ch, x / cw) with
 *       partial cells at the edges; cell id = (it * nCy + iy) * nCx + ix.
 *   Value = gamma[b, h] * c[b, h, cell(s), :] + noise[b, s, h, :] (gamma = 0 or
 *       no grid: noise only), computed in double, rounded to float, then to bf16
 *       with round-to-nearest-even.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static uint64_t splitmix64(uint64_t x)
{
    x += 0x9E3779B97F4A7C15ull;
    x = (x ^ (x >> 30)) * 0xBF58476D1CE4E5B9ull;
    x = (x ^ (x >> 27)) * 0x94D049BB133111EBull;
    return x ^ (x >> 31);
}

static uint64_t draw64(uint64_t seed, uint64_t stream, uint64_t index)
{
    return splitmix64(splitmix64(splitmix64(seed) ^ stream) ^ index);
}

static uint64_t stream_id(uint64_t tensor, uint64_t b, uint64_t h)
{
    return (tensor << 48) + (b << 24) + h;
}

static void normal_pair(uint64_t bits, double *z0, double *z1)
{
    const double two_pi = 6.283185307179586476925286766559;
    const uint32_t hi = (uint32_t)(bits >> 32), lo = (uint32_t)bits;
    const double u1 = ((double)hi + 1.0) * (1.0 / 4294967296.0);
    const double u2 = (double)lo * (1.0 / 4294967296.0);
    const double r = sqrt(-2.0 * log(u1));
    *z0 = r * cos(two_pi * u2);
    *z1 = r * sin(two_pi * u2);
}

/* One row of d standard normals (d even) for counter `row` of a stream. */
static void normal_row(uint64_t seed, uint64_t stream, uint64_t row, int d, double *out)
{
    for (int t = 0; t < d; t += 2)
        normal_pair(draw64(seed, stream, (row * (uint64_t)d + (uint64_t)t) >> 1), &out[t], &out[t + 1]);
}

/* float -> bf16 bits, round to nearest even (NaN kept quiet). */
uint16_t synth_f32_to_bf16(float f)
{
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu))
        return (uint16_t)((u >> 16) | 0x0040u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

/* A uniform double in [0, 1) for (seed, stream, index): 53 high bits of one draw. */
double synth_uniform(uint64_t seed, uint64_t stream, uint64_t index)
{
    return (double)(draw64(seed, stream, index) >> 11) * (1.0 / 9007199254740992.0);
}

/*
 * Fill rows s in [s_begin, s_end) of every (b, h) of a [B, S, H, d] bf16 tensor.
 * tensor: 1 = Q, 2 = K, 3 = V (selects the noise stream).
 * grid/cell: token grid T x Hg x W and cell ct x ch x cw; grid_t <= 0 means no
 *            grid (pure noise). S must not exceed T * Hg * W when a grid is given.
 * gamma: [B * H] centre weights, or NULL for pure noise.
 * Returns 0, or 1 on invalid arguments.
 */
int synth_fill(uint16_t *out, int tensor, uint64_t seed, int B, int S, int H, int d,
               int grid_t, int grid_h, int grid_w, int cell_t, int cell_h, int cell_w,
               const double *gamma, int s_begin, int s_end)
{
    if (!out || tensor < 1 || tensor > 3 || B <= 0 || S <= 0 || H <= 0 || d <= 0 || (d & 1) ||
        d > 1024 || s_begin < 0 || s_end > S || s_begin > s_end)
        return 1;
    const int use_grid = grid_t > 0 && gamma != NULL;
    if (use_grid && (grid_h <= 0 || grid_w <= 0 || cell_t <= 0 || cell_h <= 0 || cell_w <= 0 ||
                     (long long)grid_t * grid_h * grid_w < S))
        return 1;
    const int n_cy = use_grid ? (grid_h + cell_h - 1) / cell_h : 1;
    const int n_cx = use_grid ? (grid_w + cell_w - 1) / cell_w : 1;

    double noise[1024], centre[1024];
    for (int b = 0; b < B; ++b) {
        for (int s = s_begin; s < s_end; ++s) {
            uint64_t cell = 0;
            if (use_grid) {
                const int tt = s / (grid_h * grid_w);
                const int yy = (s / grid_w) % grid_h;
                const int xx = s % grid_w;
                cell = ((uint64_t)(tt / cell_t) * (uint64_t)n_cy + (uint64_t)(yy / cell_h)) * (uint64_t)n_cx +
                       (uint64_t)(xx / cell_w);
            }
            for (int h = 0; h < H; ++h) {
                const double g = use_grid ? gamma[b * H + h] : 0.0;
                normal_row(seed, stream_id((uint64_t)tensor, (uint64_t)b, (uint64_t)h), (uint64_t)s, d, noise);
                if (g != 0.0)
                    normal_row(seed, stream_id(0, (uint64_t)b, (uint64_t)h), cell, d, centre);
                uint16_t *dst = out + (((size_t)b * S + s) * H + h) * (size_t)d;
                for (int t = 0; t < d; ++t) {
                    const double x = g != 0.0 ? g * centre[t] + noise[t] : noise[t];
                    dst[t] = synth_f32_to_bf16((float)x);
                }
            }
        }
    }
    return 0;
}
