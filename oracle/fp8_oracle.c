/*
 * fp8_oracle.c -- plain CPU oracle for the FP8 KV-cache layout of MLA decode.
 *
 * TEST INFRASTRUCTURE ONLY (as mla_oracle.c): nothing in the product path
 * links, loads or calls this file; it shares no code with the CUDA library.
 *
 * Source: "[DeepSeek-3] FlashMLA：把 MLA 的 KV Cache 优势变成 GPU 吞吐", sec. 12
 * (FP8 KV Cache): every cached token takes 656 bytes,
 *     bytes [0, 512)    512 float8_e4m3 values: the latent (NoPE) dims 0..511
 *     bytes [512, 528)  4 fp32 scales, scale j shared by latent dims 128j..128j+127
 *     bytes [528, 656)  64 bf16 values: the RoPE dims 512..575, not quantised
 * and the kernel dequantises the latent to BF16, joins it with the BF16 RoPE
 * and runs QK and PV on BF16 inputs with FP32 accumulation.  So the FP8 path
 * computes dense MLA decode over the dequantised cache
 *     k[c]       = bf16( e4m3(latent[c]) * scale[c / 128] ),  c < 512
 *     k[512 + c] = rope[c]
 * Readings of what the page leaves open:
 *   - the regions follow each other in the order the page's table lists them;
 *   - dequantisation multiplies the e4m3 value by its scale;
 *   - "to BF16" rounds the exact product to nearest, ties to even;
 *   - e4m3 is the finite-only variant (no infinities; S.1111.111 is NaN),
 *     the float8_e4m3 of the page.
 * Here: oracle_fp8_dequant writes the bf16 bit patterns of the dequantised
 * rows; the attention itself is then the dense oracle (mla_oracle.c) on them.
 *
 * Parity status: pinned by the CPU tests (e4m3 decoding of all 256
 * codes and the bf16 rounding against torch's conversions; the whole
 * dequantisation against a torch-only restatement; power-of-two scales exact).
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

/* Value of one float8_e4m3 code: 1 sign bit, 4 exponent bits (bias 7), 3
 * mantissa bits; exponent 0 is subnormal (mantissa * 2^-9); exponent 15 with
 * mantissa 7 is NaN.  Exported for the pins. */
double oracle_e4m3_value(uint8_t code) {
    const int sign = code >> 7, e = (code >> 3) & 0xF, m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m, -9);
    else
        v = ldexp(1.0 + m / 8.0, e - 7);
    return sign ? -v : v;
}

/* bf16 bit pattern of x rounded to nearest, ties to even (8 significant bits,
 * the fp32 exponent range: normals from 2^-126, subnormals down to 2^-133,
 * overflow to infinity).  Exported for the pins. */
uint16_t oracle_bf16_round(double x) {
    uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x))
        return 0x7FC0u;
    double a = fabs(x);
    if (isinf(a))
        return sign | 0x7F80u;
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): the leading bit has weight 2^(e-1) */
    int lead = e - 1;
    if (lead < -126)
        lead = -126; /* subnormal range: fixed quantum 2^-133 */
    const double quantum = ldexp(1.0, lead - 7);
    double n = a / quantum; /* exact: a power-of-two scaling */
    double r = floor(n);
    const double frac = n - r;
    if (frac > 0.5 || (frac == 0.5 && fmod(r, 2.0) != 0.0))
        r += 1.0;
    const double v = r * quantum;
    if (v >= ldexp(1.0, 128))
        return sign | 0x7F80u;
    /* encode v (now exactly representable in bf16) through its fp32 bits */
    const float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)((u >> 16) & 0x7FFFu);
}

/*
 * oracle_fp8_dequant: rows of 656 bytes (n_tokens of them, row stride
 * row_bytes >= 656) -> bf16 bit patterns [n_tokens][576].  Returns 0, or -3
 * for bad sizes.
 */
int oracle_fp8_dequant(const uint8_t *rows, int64_t n_tokens, int64_t row_bytes, uint16_t *out) {
    if (n_tokens < 0 || row_bytes < 656)
        return -3;
    for (int64_t t = 0; t < n_tokens; ++t) {
        const uint8_t *r = rows + t * row_bytes;
        uint16_t *o = out + t * 576;
        float scale[4];
        memcpy(scale, r + 512, sizeof scale);
        for (int c = 0; c < 512; ++c)
            o[c] = oracle_bf16_round(oracle_e4m3_value(r[c]) * (double)scale[c / 128]);
        memcpy(o + 512, r + 528, 64 * sizeof(uint16_t));
    }
    return 0;
}
