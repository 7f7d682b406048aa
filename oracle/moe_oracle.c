/*
 * moe_oracle.c -- plain, slow CPU oracle of the routed NVFP4 SiTU MoE forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this file; only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant
 * generator with the CUDA library.
 *
 * Sources (web pages the method is described on):
 *   [Cake]   FlashInfer tutorial "Cake SiTU backend": the operation, the six
 *            quant_scales, qX = 1/dX and qA = 1/dA, the default SiTU
 *            (4*tanh(g/4)*sigmoid(g))*(25*tanh(u/25)), storage shapes of w13/w2
 *            and their group-16 E4M3 block scales, BF16 weighted finalize.
 *   [Ascend] torch_npu "npu_moe_init_routing_v2", section "计算公式" (formulas
 *            1-6): keyValueSort, expanded_row_idx gather/scatter, histogram,
 *            dynamic int8 quant, token move with drop/pad; parameter section for
 *            row_idx_type, expert_tokens_num_type, drop_pad_mode.
 *   [Edge]   TensorRT-Edge-LLM "Nvfp4 Tensor": global scale applied after block
 *            dequantization; 128x4 atom layout of E4M3 block scales.
 *
 * Readings where the pages are silent (listed again in the design notes):
 *   - sort is stable, ties by flat row index ascending;
 *   - cumsum is inclusive;
 *   - drop_pad keeps the lowest ranks of each expert, gather index e*C+r,
 *     unclipped histogram, unfilled slots zero;
 *   - int8 round is half-to-even with clamp to +-127, zero rows give q = 0;
 *   - NVFP4 group quant: amax -> sf = E4M3_rn_sat((amax*q)/6) -> S ->
 *     r = q/S (0 if S == 0) -> code = E2M1_rn_sat(v*r), all in fp32, no FMA;
 *   - w13 rows 0..I-1 are gate, I..2I-1 are up; low nibble is the even element.
 *
 * Floating point: dot products accumulate in fp64; every fp32 step of the
 * quantizers is written as separate fp32 operations and the file must be
 * compiled with -ffp-contract=off.
 */
#include <stdint.h>
#include <stddef.h>
#include <string.h>
#include <stdlib.h>
#include <math.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------------------ */
/* E2M1 (FP4) codec.  Values {0, .5, 1, 1.5, 2, 3, 4, 6}, sign in bit 3.      */
/* ------------------------------------------------------------------------ */

static const double kE2M1Mag[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double oracle_e2m1_value(uint8_t nib) {
    double m = kE2M1Mag[nib & 7];
    return (nib & 8) ? -m : m;
}

/* Round-to-nearest-even onto the E2M1 grid, saturating to 6.  Ties pick the
 * code with an even last bit.  The sign of the input is kept, also when the
 * magnitude rounds to zero.  NaN maps to +6 (it never occurs on valid data;
 * the page defines no NaN for E2M1). */
uint8_t oracle_e2m1_encode(float v) {
    uint8_t sign = signbit(v) ? 8 : 0;
    double a = fabs((double)v);
    uint8_t c;
    if (isnan(v)) return 7;
    if (a < 0.25) c = 0;
    else if (a == 0.25) c = 0;      /* tie 0 | 0.5   -> code 0 */
    else if (a < 0.75) c = 1;
    else if (a == 0.75) c = 2;      /* tie 0.5 | 1   -> code 2 */
    else if (a < 1.25) c = 2;
    else if (a == 1.25) c = 2;      /* tie 1 | 1.5   -> code 2 */
    else if (a < 1.75) c = 3;
    else if (a == 1.75) c = 4;      /* tie 1.5 | 2   -> code 4 */
    else if (a < 2.5) c = 4;
    else if (a == 2.5) c = 4;       /* tie 2 | 3     -> code 4 */
    else if (a < 3.5) c = 5;
    else if (a == 3.5) c = 6;       /* tie 3 | 4     -> code 6 */
    else if (a < 5.0) c = 6;
    else if (a == 5.0) c = 6;       /* tie 4 | 6     -> code 6 */
    else c = 7;                     /* above 5 and saturation */
    return (uint8_t)(sign | c);
}

/* ------------------------------------------------------------------------ */
/* E4M3 ("fn": bias 7, max 448, no inf, 0x7F/0xFF NaN) codec.                */
/* ------------------------------------------------------------------------ */

double oracle_e4m3_value(uint8_t b) {
    int s = (b >> 7) & 1, e = (b >> 3) & 15, m = b & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m, -9);              /* subnormal m * 2^-9 */
    else v = ldexp(1.0 + m / 8.0, e - 7);
    return s ? -v : v;
}

/* Round-to-nearest-even onto the E4M3 grid; magnitudes of 448 and above
 * (and infinities) saturate to 448; NaN gives 0x7F. */
uint8_t oracle_e4m3_encode(float v) {
    uint8_t sign = signbit(v) ? 0x80 : 0;
    double a = fabs((double)v);
    uint32_t code;
    if (isnan(v)) return 0x7F;
    if (a >= 448.0) return (uint8_t)(sign | 0x7E);
    if (a < ldexp(1.0, -6)) {
        /* subnormal range: grid step 2^-9 */
        double n = a / ldexp(1.0, -9);
        double fl = floor(n), fr = n - fl;
        uint32_t m = (uint32_t)fl;
        if (fr > 0.5 || (fr == 0.5 && (m & 1))) m += 1;
        code = m;                        /* m == 8 is 2^-6, the first normal */
    } else {
        int ex;
        frexp(a, &ex);                   /* a = f * 2^ex, f in [0.5, 1) */
        int e = ex - 1;                  /* a in [2^e, 2^(e+1)) */
        double n = a / ldexp(1.0, e - 3); /* in [8, 16) */
        double fl = floor(n), fr = n - fl;
        uint32_t m = (uint32_t)fl;
        if (fr > 0.5 || (fr == 0.5 && (m & 1))) m += 1;
        code = (uint32_t)(e + 7) * 8u + (m - 8u);  /* m == 16 carries */
        if (code > 0x7E) code = 0x7E;
    }
    return (uint8_t)(sign | code);
}

/* ------------------------------------------------------------------------ */
/* BF16 helpers.                                                              */
/* ------------------------------------------------------------------------ */

float oracle_bf16_to_float(uint16_t h) {
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, 4);
    return f;
}

/* fp32 -> bf16, round to nearest even (NaN kept quiet). */
uint16_t oracle_float_to_bf16(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x007FFFFFu)) return (uint16_t)((u >> 16) | 0x40);
    uint32_t lsb = (u >> 16) & 1u;
    u += 0x7FFFu + lsb;
    return (uint16_t)(u >> 16);
}

/* ------------------------------------------------------------------------ */
/* NVFP4 group-16 quantization ([Cake] group-16 NVFP4 with encode scale q;   */
/* [Edge] global scale applied after block dequantization).                  */
/* ------------------------------------------------------------------------ */

/* Quantize one group of 16 fp32 values with encode scale q.
 * codes16[j] receives the 4-bit code of element j (one code per byte);
 * *sf receives the E4M3 block scale byte. */
void oracle_nvfp4_quant_group(const float* v, float q, uint8_t* codes16, uint8_t* sf) {
    float amax = 0.0f;
    for (int j = 0; j < 16; ++j) {
        float a = fabsf(v[j]);
        if (a > amax) amax = a;
    }
    float t = amax * q;
    float t6 = t / 6.0f;
    uint8_t s = oracle_e4m3_encode(t6);
    float S = (float)oracle_e4m3_value(s);
    float r = (S == 0.0f) ? 0.0f : q / S;
    for (int j = 0; j < 16; ++j) {
        float y = v[j] * r;
        codes16[j] = oracle_e2m1_encode(y);
    }
    *sf = s;
}

/* Quantize rows x cols fp32 (cols % 16 == 0) with one encode scale per row
 * (q_per_row != NULL) or a single scale q.  Output is the canonical layout:
 * packed codes [rows, cols/2] (even element in the low nibble) and row-major
 * scales [rows, cols/16]. */
void oracle_nvfp4_quant_rows(const float* x, int64_t rows, int64_t cols,
                             const float* q_per_row, float q,
                             uint8_t* packed, uint8_t* sf) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        float qq = q_per_row ? q_per_row[r] : q;
        uint8_t codes[16];
        for (int64_t g = 0; g < cols / 16; ++g) {
            oracle_nvfp4_quant_group(x + r * cols + g * 16, qq, codes, &sf[r * (cols / 16) + g]);
            for (int j = 0; j < 8; ++j)
                packed[r * (cols / 2) + g * 8 + j] = (uint8_t)(codes[2 * j] | (codes[2 * j + 1] << 4));
        }
    }
}

/* Dequantize canonical packed codes and block scales to fp64 values
 * E2M1(code) * S (the global scale is applied separately). */
void oracle_nvfp4_dequant_rows(const uint8_t* packed, const uint8_t* sf, int64_t rows, int64_t cols,
                               double* out) {
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t c = 0; c < cols; ++c) {
            uint8_t b = packed[r * (cols / 2) + c / 2];
            uint8_t nib = (c & 1) ? (b >> 4) : (b & 15);
            out[r * cols + c] = oracle_e2m1_value(nib) * oracle_e4m3_value(sf[r * (cols / 16) + c / 16]);
        }
}

/* ------------------------------------------------------------------------ */
/* Routing ([Ascend] formulas 1-3).                                           */
/* ------------------------------------------------------------------------ */

/* keyValueSort(expertIdx, rowIdx) with rowIdx = t*k + j, stable.  Written as
 * the plain two-loop counting form: experts in ascending order, and within
 * one expert the flat indices in ascending order.  Ids outside [0, E) are not
 * routed: they take no sorted position and their gather entry is -1.
 *   sorted_row[i]          scatter form, expandedRowIdx[i] = sortedRowIdx[i]
 *   gather[sorted_row[i]]  gather form,  = i
 *   count[e]               histogram of sortedExpertIdx
 *   cumsum[e]              inclusive prefix sum of count
 * Returns the number of routed (valid) pairs. */
int64_t oracle_routing(const int32_t* ids, int64_t T, int32_t k, int32_t E,
                       int32_t* sorted_row, int32_t* sorted_expert, int32_t* gather,
                       int32_t* count, int32_t* cumsum) {
    int64_t P = T * (int64_t)k;
    for (int64_t f = 0; f < P; ++f) gather[f] = -1;
    int64_t i = 0;
    for (int32_t e = 0; e < E; ++e) {
        int32_t c = 0;
        for (int64_t f = 0; f < P; ++f) {
            if (ids[f] == e) {
                sorted_row[i] = (int32_t)f;
                if (sorted_expert) sorted_expert[i] = e;
                gather[f] = (int32_t)i;
                ++i;
                ++c;
            }
        }
        count[e] = c;
        cumsum[e] = (int32_t)i;
    }
    for (int64_t r = i; r < P; ++r) {
        sorted_row[r] = -1;
        if (sorted_expert) sorted_expert[r] = -1;
    }
    return i;
}

/* ------------------------------------------------------------------------ */
/* Init-routing token move with optional dynamic int8 quant and drop/pad     */
/* ([Ascend] formulas 4-5 and the drop_pad_mode / expert_capacity params).   */
/* ------------------------------------------------------------------------ */

/* Dynamic int8 row quant: s = row_max(|x|)/127, q = round(x/s). */
void oracle_dynamic_int8_row(const uint16_t* xbf, int64_t H, int8_t* q, float* scale) {
    float amax = 0.0f;
    for (int64_t h = 0; h < H; ++h) {
        float a = fabsf(oracle_bf16_to_float(xbf[h]));
        if (a > amax) amax = a;
    }
    float s = amax / 127.0f;
    for (int64_t h = 0; h < H; ++h) {
        if (s == 0.0f) { q[h] = 0; continue; }
        float y = oracle_bf16_to_float(xbf[h]) / s;
        float rr = nearbyintf(y);            /* default rounding mode: half to even */
        if (rr > 127.0f) rr = 127.0f;
        if (rr < -127.0f) rr = -127.0f;
        q[h] = (int8_t)rr;
    }
    *scale = s;
}

/* Full init-routing.
 *   drop_pad          0 dropless (expanded rows = valid pairs in sorted order),
 *                     1 drop/pad to [E, C, H]
 *   row_idx_type      0 gather form, 1 scatter form
 *   tokens_num_type   0 inclusive cumsum, 1 count
 *   quant_mode        -1 none (expanded_x is bf16), 1 dynamic int8
 * expanded_x: dropless [P, H] (rows beyond the valid count untouched),
 *             drop_pad [E*C, H] (unfilled slots zero)
 * expanded_scale: one fp32 per expanded row (quant_mode 1 only; unfilled 0)
 * expanded_row_idx: [P]
 * Returns the number of valid pairs. */
int64_t oracle_init_routing(const uint16_t* x, const int32_t* ids, int64_t T, int32_t k, int32_t E,
                            int64_t H, int32_t drop_pad, int32_t C, int32_t row_idx_type,
                            int32_t tokens_num_type, int32_t quant_mode,
                            void* expanded_x, int32_t* expanded_row_idx,
                            int32_t* tokens_out, float* expanded_scale) {
    int64_t P = T * (int64_t)k;
    int32_t* sorted_row = (int32_t*)malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
    int32_t* sorted_expert = (int32_t*)malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
    int32_t* gather = (int32_t*)malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
    int32_t* count = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    int32_t* cumsum = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    int64_t nvalid = oracle_routing(ids, T, k, E, sorted_row, sorted_expert, gather, count, cumsum);

    /* per-token quant (or copy) once; the move then takes rows by index */
    int8_t* qx = NULL;
    float* qs = NULL;
    if (quant_mode == 1) {
        qx = (int8_t*)malloc((size_t)(T * H > 0 ? T * H : 1));
        qs = (float*)malloc(sizeof(float) * (size_t)(T > 0 ? T : 1));
        for (int64_t t = 0; t < T; ++t) oracle_dynamic_int8_row(x + t * H, H, qx + t * H, &qs[t]);
    }
    size_t esz = (quant_mode == 1) ? 1 : 2;

    /* destination row of sorted position i */
    int32_t* dest = (int32_t*)malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
    for (int64_t i = 0; i < nvalid; ++i) {
        if (!drop_pad) {
            dest[i] = (int32_t)i;
        } else {
            int32_t e = sorted_expert[i];
            int64_t off = cumsum[e] - count[e];
            int64_t r = i - off;
            dest[i] = (r < C) ? (int32_t)(e * (int64_t)C + r) : -1;
        }
    }
    if (drop_pad) {
        memset(expanded_x, 0, (size_t)E * (size_t)C * (size_t)H * esz);
        if (expanded_scale) memset(expanded_scale, 0, sizeof(float) * (size_t)E * (size_t)C);
    }
    for (int64_t i = 0; i < nvalid; ++i) {
        if (dest[i] < 0) continue;
        int64_t t = sorted_row[i] / k;
        if (quant_mode == 1) {
            memcpy((int8_t*)expanded_x + (int64_t)dest[i] * H, qx + t * H, (size_t)H);
            if (expanded_scale) expanded_scale[dest[i]] = qs[t];
        } else {
            memcpy((uint16_t*)expanded_x + (int64_t)dest[i] * H, x + t * H, (size_t)H * 2);
        }
    }
    /* expanded_row_idx */
    if (row_idx_type == 1) {
        for (int64_t i = 0; i < P; ++i) expanded_row_idx[i] = sorted_row[i];
    } else {
        for (int64_t f = 0; f < P; ++f) expanded_row_idx[f] = -1;
        for (int64_t i = 0; i < nvalid; ++i) expanded_row_idx[sorted_row[i]] = dest[i];
    }
    for (int32_t e = 0; e < E; ++e) tokens_out[e] = (tokens_num_type == 1) ? count[e] : cumsum[e];

    free(dest); free(qx); free(qs);
    free(sorted_row); free(sorted_expert); free(gather); free(count); free(cumsum);
    return nvalid;
}

/* Init-routing with every option of the page's parameter list ([Ascend]
 * formulas 1-6 and the parameters active_expert_range, active_num,
 * expert_tokens_num_type, quant_mode, scale, offset).  Readings where the
 * page is loose are marked (r).
 *   expert_start, expert_end   active range [start, end) of expert ids; pairs
 *                              whose id lies outside it are not routed (ids
 *                              outside [0, E) are not routed either)
 *   active_num                 > 0: only the first min(active_num, available)
 *                              sorted rows are moved (Active); <= 0 dropless
 *   drop_pad, C                as in oracle_init_routing (full range only)
 *   row_idx_type               0 gather form, 1 scatter form
 *   tokens_num_type            0 inclusive cumsum, 1 count, over the range
 *                              (end-start entries); 2 key_value: rows
 *                              (expert id, count) of the in-range experts
 *                              with a non-zero count, in expert order, at the
 *                              head of [E, 2]; the remaining rows 0 (r)
 *   quant_mode -1              bf16 copy; scale [T] or NULL: expanded_scale
 *                              of a row = scale of its token
 *   quant_mode 0 (static)      q = rint(x*scale[0] + offset[0]) in fp32, half
 *                              to even, saturated to [-128, 127] (r); no
 *                              expanded_scale
 *   quant_mode 1 (dynamic)     smooth = scale [nsr, H] or NULL (nsr 1 or
 *                              end-start): xs = x * smooth[row of the pair's
 *                              expert - start, or 0]; s = row_max|xs|/127;
 *                              q = rint(xs / s) clamped to +-127 (r: the
 *                              page's quotient omits the smooth factor, which
 *                              it used to compute s); expanded_scale = s
 * expanded_row_idx gather form: the moved row of a pair, else -1; scatter
 * form: sorted_row for the available pairs, then -1.
 * Returns availableIdxNum, the number of pairs with an id in the range. */
int64_t oracle_init_routing_ex(const uint16_t* x, const int32_t* ids, int64_t T, int32_t k, int32_t E, int64_t H,
                               int32_t expert_start, int32_t expert_end, int64_t active_num, int32_t drop_pad,
                               int32_t C, int32_t row_idx_type, int32_t tokens_num_type, int32_t quant_mode,
                               const float* scale, int32_t scale_rows, const float* offset, void* expanded_x,
                               int32_t* expanded_row_idx, int32_t* tokens_out, float* expanded_scale) {
    int64_t P = T * (int64_t)k;
    int32_t R = expert_end - expert_start;
    int32_t* sorted_row = (int32_t*)malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
    int32_t* sorted_expert = (int32_t*)malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
    int32_t* count = (int32_t*)calloc((size_t)(R > 0 ? R : 1), sizeof(int32_t));
    int32_t* cumsum = (int32_t*)calloc((size_t)(R > 0 ? R : 1), sizeof(int32_t));
    /* formulas 1 and 3 over the active range: stable by (expert, flat index) */
    int64_t avail = 0;
    for (int32_t e = expert_start; e < expert_end; ++e) {
        for (int64_t f = 0; f < P; ++f)
            if (ids[f] == e) {
                sorted_row[avail] = (int32_t)f;
                sorted_expert[avail] = e;
                ++avail;
                ++count[e - expert_start];
            }
        cumsum[e - expert_start] = (int32_t)avail;
    }
    int64_t nmove = (active_num > 0 && active_num < avail) ? active_num : avail;
    size_t esz = (quant_mode == -1) ? 2 : 1;
    /* destination row of sorted position i */
    int32_t* dest = (int32_t*)malloc(sizeof(int32_t) * (size_t)(P > 0 ? P : 1));
    for (int64_t i = 0; i < avail; ++i) {
        if (!drop_pad) {
            dest[i] = (i < nmove) ? (int32_t)i : -1;
        } else {
            int32_t e = sorted_expert[i] - expert_start;
            int64_t r = i - (cumsum[e] - count[e]);
            dest[i] = (r < C) ? (int32_t)(e * (int64_t)C + r) : -1;
        }
    }
    if (drop_pad) {
        memset(expanded_x, 0, (size_t)R * (size_t)C * (size_t)H * esz);
        if (expanded_scale) memset(expanded_scale, 0, sizeof(float) * (size_t)R * (size_t)C);
    }
    /* formulas 4 and 5, one moved row at a time */
    float* xs = (float*)malloc(sizeof(float) * (size_t)(H > 0 ? H : 1));
    for (int64_t i = 0; i < avail; ++i) {
        if (dest[i] < 0) continue;
        int64_t t = sorted_row[i] / k;
        const uint16_t* xr = x + t * H;
        if (quant_mode == -1) {
            memcpy((uint16_t*)expanded_x + (int64_t)dest[i] * H, xr, (size_t)H * 2);
            if (expanded_scale && scale) expanded_scale[dest[i]] = scale[t];
        } else if (quant_mode == 0) {
            int8_t* q = (int8_t*)expanded_x + (int64_t)dest[i] * H;
            for (int64_t h = 0; h < H; ++h) {
                float v = oracle_bf16_to_float(xr[h]) * scale[0];
                v = v + offset[0];
                float rr = nearbyintf(v);
                if (rr > 127.0f) rr = 127.0f;
                if (rr < -128.0f) rr = -128.0f;
                q[h] = (int8_t)rr;
            }
        } else {
            const float* sm = NULL;
            if (scale && scale_rows > 0) sm = scale + (scale_rows == 1 ? 0 : (int64_t)(sorted_expert[i] - expert_start)) * H;
            float amax = 0.0f;
            for (int64_t h = 0; h < H; ++h) {
                float v = oracle_bf16_to_float(xr[h]);
                if (sm) v = v * sm[h];
                xs[h] = v;
                if (fabsf(v) > amax) amax = fabsf(v);
            }
            float sc = amax / 127.0f;
            int8_t* q = (int8_t*)expanded_x + (int64_t)dest[i] * H;
            for (int64_t h = 0; h < H; ++h) {
                if (sc == 0.0f) { q[h] = 0; continue; }
                float rr = nearbyintf(xs[h] / sc);
                if (rr > 127.0f) rr = 127.0f;
                if (rr < -127.0f) rr = -127.0f;
                q[h] = (int8_t)rr;
            }
            if (expanded_scale) expanded_scale[dest[i]] = sc;
        }
    }
    /* formula 2 */
    if (row_idx_type == 1) {
        for (int64_t i = 0; i < P; ++i) expanded_row_idx[i] = (i < avail) ? sorted_row[i] : -1;
    } else {
        for (int64_t f = 0; f < P; ++f) expanded_row_idx[f] = -1;
        for (int64_t i = 0; i < avail; ++i) expanded_row_idx[sorted_row[i]] = dest[i];
    }
    /* formula 3 output */
    if (tokens_num_type == 2) {
        for (int64_t j = 0; j < 2 * (int64_t)E; ++j) tokens_out[j] = 0;
        int64_t n = 0;
        for (int32_t e = 0; e < R; ++e)
            if (count[e] > 0) {
                tokens_out[2 * n] = expert_start + e;
                tokens_out[2 * n + 1] = count[e];
                ++n;
            }
    } else {
        for (int32_t e = 0; e < R; ++e) tokens_out[e] = (tokens_num_type == 1) ? count[e] : cumsum[e];
    }
    free(xs); free(dest); free(sorted_row); free(sorted_expert); free(count); free(cumsum);
    return avail;
}

/* ------------------------------------------------------------------------ */
/* SiTU ([Cake] "Default SiTU is (4*tanh(g/4)*sigmoid(g))*(25*tanh(u/25))",  */
/* per-expert beta / linear beta optional).                                   */
/* ------------------------------------------------------------------------ */

double oracle_situ(double g, double u, double beta, double lam) {
    double gate = beta * tanh(g / beta) * (1.0 / (1.0 + exp(-g)));
    double lin = lam * tanh(u / lam);
    return gate * lin;
}

/* ------------------------------------------------------------------------ */
/* MoE forward for a list of tokens ([Cake]: quant X, FC1, SiTU, requant,     */
/* FC2, BF16 weighted finalize).  Weights in the canonical layout:            */
/*   w13 [E, 2I, H/2] packed E2M1, sf13 [E, 2I, H/16] E4M3 (gate rows first) */
/*   w2  [E, H, I/2],               sf2  [E, H, I/16]                        */
/* The six scales: qX[1], dXdW13[E], qA[E], dAdW2[E] (block scales are the   */
/* sf arrays).  beta/lam may be NULL (defaults 4 and 25).                     */
/* Outputs (any may be NULL):                                                 */
/*   out[ntok, H] bf16; z_out[ntok, k, 2I] fp32 FC1 pre-activations;          */
/*   a_out[ntok, k, I] fp32 SiTU outputs; aq_out[ntok, k, I/2] packed codes;   */
/*   asf_out[ntok, k, I/16] E4M3; y_out[ntok, k, H] fp32 FC2 outputs.          */
/* ------------------------------------------------------------------------ */

void oracle_moe_forward_tokens(int32_t H, int32_t I, int32_t E, int32_t k,
                               const uint16_t* x, const int32_t* ids, const uint16_t* route_w,
                               const int64_t* tokens, int64_t ntok,
                               const uint8_t* w13, const uint8_t* sf13,
                               const uint8_t* w2, const uint8_t* sf2,
                               const float* qX, const float* dXdW13, const float* qA,
                               const float* dAdW2, const float* beta, const float* lam,
                               uint16_t* out, float* z_out, float* a_out,
                               uint8_t* aq_out, uint8_t* asf_out, float* y_out) {
    const int64_t twoI = 2 * (int64_t)I;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t ti = 0; ti < ntok; ++ti) {
        int64_t t = tokens[ti];
        /* 1. quantize the token row with qX */
        float* xf = (float*)malloc(sizeof(float) * (size_t)H);
        uint8_t* xc = (uint8_t*)malloc((size_t)H);
        uint8_t* xs = (uint8_t*)malloc((size_t)H / 16);
        double* xd = (double*)malloc(sizeof(double) * (size_t)H);
        for (int64_t h = 0; h < H; ++h) xf[h] = oracle_bf16_to_float(x[t * H + h]);
        for (int64_t g = 0; g < H / 16; ++g) oracle_nvfp4_quant_group(xf + g * 16, qX[0], xc + g * 16, &xs[g]);
        for (int64_t h = 0; h < H; ++h) xd[h] = oracle_e2m1_value(xc[h]) * oracle_e4m3_value(xs[h / 16]);

        double* acc_out = (double*)calloc((size_t)H, sizeof(double));
        float* z = (float*)malloc(sizeof(float) * (size_t)twoI);
        float* a = (float*)malloc(sizeof(float) * (size_t)I);
        uint8_t* ac = (uint8_t*)malloc((size_t)I);
        uint8_t* as = (uint8_t*)malloc((size_t)I / 16);
        double* ad = (double*)malloc(sizeof(double) * (size_t)I);

        for (int32_t j = 0; j < k; ++j) {
            int32_t e = ids[t * k + j];
            if (e < 0 || e >= E) continue;           /* not routed */
            /* 2. FC1: acc[n] = sum_h xhat_h * what[e,n,h]; z = float(acc) * dX*dW13[e] */
            for (int64_t n = 0; n < twoI; ++n) {
                const uint8_t* wr = w13 + ((int64_t)e * twoI + n) * (H / 2);
                const uint8_t* sr = sf13 + ((int64_t)e * twoI + n) * (H / 16);
                double acc = 0.0;
                for (int64_t h = 0; h < H; ++h) {
                    uint8_t b = wr[h / 2];
                    uint8_t nib = (h & 1) ? (b >> 4) : (b & 15);
                    double wv = oracle_e2m1_value(nib) * oracle_e4m3_value(sr[h / 16]);
                    acc += xd[h] * wv;
                }
                float af = (float)acc;
                z[n] = af * dXdW13[e];
            }
            /* 3. SiTU on (g, u) = (z[0:I], z[I:2I]) in fp64, rounded to fp32 */
            double be = beta ? (double)beta[e] : 4.0;
            double la = lam ? (double)lam[e] : 25.0;
            for (int64_t i = 0; i < I; ++i) a[i] = (float)oracle_situ((double)z[i], (double)z[I + i], be, la);
            /* 4. requant with qA[e] */
            for (int64_t g = 0; g < I / 16; ++g) oracle_nvfp4_quant_group(a + g * 16, qA[e], ac + g * 16, &as[g]);
            for (int64_t i = 0; i < I; ++i) ad[i] = oracle_e2m1_value(ac[i]) * oracle_e4m3_value(as[i / 16]);
            /* 5. FC2: y[h] = float(sum_i ahat_i * w2hat[e,h,i]) * dA*dW2[e]; 6. weight and sum */
            double wt = (double)oracle_bf16_to_float(route_w[t * k + j]);
            for (int64_t h = 0; h < H; ++h) {
                const uint8_t* wr = w2 + ((int64_t)e * H + h) * (I / 2);
                const uint8_t* sr = sf2 + ((int64_t)e * H + h) * (I / 16);
                double acc = 0.0;
                for (int64_t i = 0; i < I; ++i) {
                    uint8_t b = wr[i / 2];
                    uint8_t nib = (i & 1) ? (b >> 4) : (b & 15);
                    acc += ad[i] * (oracle_e2m1_value(nib) * oracle_e4m3_value(sr[i / 16]));
                }
                float yf = (float)acc;
                float y = yf * dAdW2[e];
                if (y_out) y_out[(ti * k + j) * (int64_t)H + h] = y;
                acc_out[h] += wt * (double)y;
            }
            if (z_out) memcpy(z_out + (ti * k + j) * twoI, z, sizeof(float) * (size_t)twoI);
            if (a_out) memcpy(a_out + (ti * k + j) * (int64_t)I, a, sizeof(float) * (size_t)I);
            if (aq_out)
                for (int64_t i = 0; i < I / 2; ++i)
                    aq_out[(ti * k + j) * (int64_t)(I / 2) + i] = (uint8_t)(ac[2 * i] | (ac[2 * i + 1] << 4));
            if (asf_out) memcpy(asf_out + (ti * k + j) * (int64_t)(I / 16), as, (size_t)I / 16);
        }
        /* 7. BF16 finalize of the fp64 k-sum (rounded through fp32) */
        if (out)
            for (int64_t h = 0; h < H; ++h) out[ti * H + h] = oracle_float_to_bf16((float)acc_out[h]);
        free(xf); free(xc); free(xs); free(xd); free(acc_out);
        free(z); free(a); free(ac); free(as); free(ad);
    }
}

/* SiTU + requant of given fp32 pre-activations (rows of [g | u], 2I wide) with
 * one expert's constants; used to check the activation stage in isolation. */
void oracle_situ_requant_rows(const float* z, int64_t rows, int32_t I, float qA, float beta, float lam,
                              float* a_out, uint8_t* packed, uint8_t* sf) {
    for (int64_t r = 0; r < rows; ++r) {
        float* a = a_out + r * I;
        for (int64_t i = 0; i < I; ++i)
            a[i] = (float)oracle_situ((double)z[r * 2 * I + i], (double)z[r * 2 * I + I + i], beta, lam);
        uint8_t codes[16];
        for (int64_t g = 0; g < I / 16; ++g) {
            oracle_nvfp4_quant_group(a + g * 16, qA, codes, &sf[r * (I / 16) + g]);
            for (int j = 0; j < 8; ++j)
                packed[r * (I / 2) + g * 8 + j] = (uint8_t)(codes[2 * j] | (codes[2 * j + 1] << 4));
        }
    }
}

/* Codec sweeps over a contiguous range of fp32 bit patterns (for exhaustive
 * checks): out[i] = encode(bits_as_float(start + i)). */
void oracle_e2m1_encode_range(uint32_t start, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = start + (uint32_t)i;
        float f;
        memcpy(&f, &u, 4);
        out[i] = oracle_e2m1_encode(f);
    }
}

void oracle_e4m3_encode_range(uint32_t start, int64_t n, uint8_t* out) {
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t u = start + (uint32_t)i;
        float f;
        memcpy(&f, &u, 4);
        out[i] = oracle_e4m3_encode(f);
    }
}

/* Byte offset of the E4M3 block scale of (mRow, kChunk) in the 128x4 atom
 * layout ("Nvfp4 Tensor", block_scale: innerK = kChunk%4, innerM =
 * (mRow%128)/32, outerM = mRow%32, kTile = kChunk/4, mTile = mRow/128,
 * offset = mTile*numKTiles*512 + kTile*512 + outerM*16 + innerM*4 + innerK),
 * with numKTiles = ceil(numSfCols/4). */
int64_t oracle_scale_atom_offset(int64_t mRow, int64_t kChunk, int64_t numSfCols) {
    int64_t numKTiles = (numSfCols + 3) / 4;
    int64_t innerK = kChunk % 4, innerM = (mRow % 128) / 32, outerM = mRow % 32;
    int64_t kTile = kChunk / 4, mTile = mRow / 128;
    return mTile * numKTiles * 512 + kTile * 512 + outerM * 16 + innerM * 4 + innerK;
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Threads used by the parallel loops from here on (the CPU baseline times the
 * oracle on all host cores and on one). */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}
