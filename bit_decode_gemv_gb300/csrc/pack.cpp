// pack.cpp -- host side of libtg: status strings, layouts and the weight packer.
//
// The packer turns host trits into the device layouts described in tg.h:
//  * ternary rows as the W_nonzero / W_negative bitmask pair (BitState brief
//    §4), two bits per weight, interleaved so that one 32-bit word yields four
//    lanes per byte-masked extract and one warp reads 512 contiguous bytes;
//  * binary Q1_0 rows (integer_engine.md §4.1) as one sign bit per weight,
//    interleaved the same way (one 16-byte chunk per row and group);
//  * the 8 base-3 planes of the lm_head (SKaiNET issue #337, BITNET_PLANES)
//    as two balanced base-3 digit groups of four planes, one byte per weight
//    each, plus the row's own bound on the planes 4-7 residual.
// Rows are split across host threads; the output does not depend on the
// thread count.

#include <algorithm>
#include <cstdint>
#include <cstring>
#include <thread>
#include <vector>

#include "tg.h"
#include "tg_internal.h"

namespace {

constexpr int64_t kAlign = 256;

int64_t align_up(int64_t v) { return (v + kAlign - 1) / kAlign * kAlign; }

template <class F>
void parallel_rows(int64_t n, F fn)
{
    unsigned hw = std::thread::hardware_concurrency();
    int64_t nt = std::max<int64_t>(1, std::min<int64_t>(hw ? hw : 1, 32));
    if (n < 256)
        nt = 1;
    nt = std::min(nt, n);
    if (nt <= 1) {
        fn(0, n);
        return;
    }
    std::vector<std::thread> pool;
    int64_t per = (n + nt - 1) / nt;
    for (int64_t t = 0; t < nt; t++) {
        int64_t a = t * per, b = std::min(n, a + per);
        if (a < b)
            pool.emplace_back(fn, a, b);
    }
    for (auto &th : pool)
        th.join();
}

void store_u32(uint8_t *p, uint32_t v)
{
    p[0] = (uint8_t)(v & 0xff);
    p[1] = (uint8_t)((v >> 8) & 0xff);
    p[2] = (uint8_t)((v >> 16) & 0xff);
    p[3] = (uint8_t)((v >> 24) & 0xff);
}

}  // namespace

extern "C" const char *tg_status_string(int status)
{
    switch (status) {
    case TG_OK: return "ok";
    case TG_ERR_ARG: return "invalid argument (null or misaligned pointer, unknown kind, wrong layout)";
    case TG_ERR_SHAPE: return "invalid shape (N, K, M or k out of range)";
    case TG_ERR_VALUE: return "invalid value (trit outside {-1,0,1}, binary weight not -1/+1, or row scale <= 0)";
    case TG_ERR_BOUND: return "integer bound exceeded: a worst-case sum could overflow";
    case TG_ERR_WORKSPACE: return "workspace or output buffer missing, misaligned or too small";
    case TG_ERR_CUDA: return "CUDA error";
    case TG_ERR_DEVICE: return "a kernel gave up a bounded wait";
    default: return "unknown status";
    }
}

extern "C" int tg_layout_init(int kind, int64_t N, int64_t K, tg_layout *out)
{
    if (!out)
        return TG_ERR_ARG;
    if (kind != TG_TERNARY_I8 && kind != TG_TERNARY_LNS8 && kind != TG_PLANES8 && kind != TG_BINARY_Q1)
        return TG_ERR_ARG;
    if (N < 1 || K < TG_GROUP || K % TG_GROUP != 0 || N > ((int64_t)1 << 31) - 1 ||
        K > ((int64_t)1 << 24))
        return TG_ERR_SHAPE;
    tg_layout L;
    std::memset(&L, 0, sizeof(L));
    L.kind = kind;
    L.version = 1;
    L.N = N;
    L.K = K;
    L.G = K / TG_GROUP;
    if (kind == TG_PLANES8) {
        // rows of 2K bytes: planes 0-3 (K bytes) then planes 4-7 (K bytes)
        L.tiles = 0;
        L.mask_off = 0;
        L.mask_bytes = N * K;
        L.aux_off = K;
        L.aux_bytes = N * K;
        L.scale_off = align_up(2 * N * K);
        L.scale_bytes = N * 4;
        L.aux2_off = align_up(L.scale_off + L.scale_bytes);
        L.aux2_bytes = N;
        L.total_bytes = align_up(L.aux2_off + L.aux2_bytes);
    } else if (kind == TG_TERNARY_I8 || kind == TG_BINARY_Q1) {
        L.tiles = (N + tgi::kTileRows - 1) / tgi::kTileRows;
        L.mask_off = 0;
        L.mask_bytes = L.tiles * L.G * tgi::kTileRows * (kind == TG_BINARY_Q1 ? 16 : 32);
        L.scale_off = align_up(L.mask_bytes);
        L.scale_bytes = L.tiles * L.G * tgi::kTileRows * 4;
        L.total_bytes = align_up(L.scale_off + L.scale_bytes);
    } else {
        // LNS8: blocks of 16 rows, the masks in tensor-core fragment order
        L.tiles = (N + tgi::kLnsBlockRows - 1) / tgi::kLnsBlockRows;
        L.mask_off = 0;
        L.mask_bytes = L.tiles * L.G * 32 * 16;
        L.scale_off = align_up(L.mask_bytes);
        L.scale_bytes = L.tiles * L.G * tgi::kLnsBlockRows;
        L.total_bytes = align_up(L.scale_off + L.scale_bytes);
    }
    *out = L;
    return TG_OK;
}

extern "C" size_t tg_packed_bytes(int kind, int64_t N, int64_t K)
{
    tg_layout L;
    if (tg_layout_init(kind, N, K, &L) != TG_OK)
        return 0;
    return (size_t)L.total_bytes;
}

namespace {

// Two-bit field of one weight: bit 0 = W_nonzero, bit 1 = W_negative.
inline uint32_t mask_field(int8_t v) { return (uint32_t)(v != 0) | ((uint32_t)(v < 0) << 1); }

// Pack ternary rows [N][K] into the tiled mask layout; returns false on a bad trit.
bool pack_masks(const tg_layout &L, const int8_t *t, uint8_t *out)
{
    const int64_t N = L.N, K = L.K, G = L.G;
    std::vector<char> bad((size_t)L.tiles, 0);
    parallel_rows(L.tiles, [&](int64_t t0, int64_t t1) {
        for (int64_t T = t0; T < t1; T++) {
            for (int64_t g = 0; g < G; g++) {
                uint8_t *blk = out + L.mask_off + (T * G + g) * 1024;
                for (int h = 0; h < 2; h++) {
                    for (int l = 0; l < tgi::kTileRows; l++) {
                        const int64_t r = T * tgi::kTileRows + l;
                        uint8_t *chunk = blk + (h * 32 + l) * 16;
                        for (int u = 0; u < 4; u++) {
                            uint32_t word = 0;
                            if (r < N) {
                                const int8_t *src = t + r * K + g * TG_GROUP + h * 64 + u * 16;
                                for (int j = 0; j < 4; j++) {
                                    for (int b = 0; b < 4; b++) {
                                        int8_t v = src[4 * j + b];
                                        if (v < -1 || v > 1)
                                            bad[(size_t)T] = 1;
                                        word |= mask_field(v) << (8 * b + 2 * j);
                                    }
                                }
                            }
                            store_u32(chunk + 4 * u, word);
                        }
                    }
                }
            }
        }
    });
    for (char b : bad)
        if (b)
            return false;
    return true;
}

// Pack binary rows [N][K] (every value -1 or +1) into the Q1 layout (tg.h):
// per (tile, group), lane l's 16 bytes are four words; word u holds group
// lanes 32u + 4j + b in bit 8b + j, set for +1. False on a value other than
// -1 or +1.
bool pack_q1(const tg_layout &L, const int8_t *t, uint8_t *out)
{
    const int64_t N = L.N, K = L.K, G = L.G;
    std::vector<char> bad((size_t)L.tiles, 0);
    parallel_rows(L.tiles, [&](int64_t t0, int64_t t1) {
        for (int64_t T = t0; T < t1; T++) {
            for (int64_t g = 0; g < G; g++) {
                uint8_t *blk = out + L.mask_off + (T * G + g) * 512;
                for (int l = 0; l < tgi::kTileRows; l++) {
                    const int64_t r = T * tgi::kTileRows + l;
                    for (int u = 0; u < 4; u++) {
                        uint32_t word = 0;
                        if (r < N) {
                            const int8_t *src = t + r * K + g * TG_GROUP + u * 32;
                            for (int j = 0; j < 8; j++) {
                                for (int b = 0; b < 4; b++) {
                                    const int8_t v = src[4 * j + b];
                                    if (v != 1 && v != -1)
                                        bad[(size_t)T] = 1;
                                    word |= (uint32_t)(v == 1) << (8 * b + j);
                                }
                            }
                        }
                        store_u32(blk + l * 16 + 4 * u, word);
                    }
                }
            }
        }
    });
    for (char b : bad)
        if (b)
            return false;
    return true;
}

// Pack ternary rows [N][K] into the LNS8 fragment layout (tg.h); false on a bad trit.
// Lane l = 4g + t of a warp holds, for each 16-lane chunk c of a group, the
// eight trits of one 16 x 16 A fragment: rows g and g+8 of the 16-row block at
// group lanes 16c + {2t, 2t+1, 2t+8, 2t+9}. Register r of chunk c (r' = 4(c%2)
// + r in word c/2) takes its low trit's W_nonzero / W_negative bits at 7 - r'
// and 15 - r', its high trit's at 23 - r' and 31 - r'.
bool pack_lns8_fragments(const tg_layout &L, const int8_t *t, uint8_t *out)
{
    const int64_t N = L.N, K = L.K, G = L.G;
    std::vector<char> bad((size_t)L.tiles, 0);
    parallel_rows(L.tiles, [&](int64_t b0, int64_t b1) {
        for (int64_t B = b0; B < b1; B++) {
            for (int64_t g = 0; g < G; g++) {
                for (int lane = 0; lane < 32; lane++) {
                    const int gq = lane >> 2, tq = lane & 3;
                    uint32_t words[4] = {0, 0, 0, 0};
                    for (int c = 0; c < 8; c++) {
                        for (int r = 0; r < 4; r++) {
                            const int row = gq + ((r & 1) ? 8 : 0);
                            const int col = 16 * c + 2 * tq + ((r & 2) ? 8 : 0);
                            const int rp = 4 * (c & 1) + r;
                            const int64_t grow = B * tgi::kLnsBlockRows + row;
                            for (int h = 0; h < 2; h++) {
                                int8_t v = 0;
                                if (grow < N) {
                                    v = t[grow * K + g * TG_GROUP + col + h];
                                    if (v < -1 || v > 1)
                                        bad[(size_t)B] = 1;
                                }
                                const uint32_t nz = v != 0, neg = v < 0;
                                words[c >> 1] |= nz << (16 * h + 7 - rp);
                                words[c >> 1] |= neg << (16 * h + 15 - rp);
                            }
                        }
                    }
                    uint8_t *dst = out + L.mask_off + ((B * G + g) * 32 + lane) * 16;
                    for (int u = 0; u < 4; u++)
                        store_u32(dst + 4 * u, words[u]);
                }
            }
        }
    });
    for (char b : bad)
        if (b)
            return false;
    return true;
}

}  // namespace

extern "C" int tg_pack_weights(int kind, int64_t N, int64_t K, const int8_t *trits,
                               const void *scales, void *out_v, size_t out_bytes, tg_layout *layout)
{
    if (!trits || !scales || !out_v || !layout)
        return TG_ERR_ARG;
    tg_layout L;
    int st = tg_layout_init(kind, N, K, &L);
    if (st != TG_OK)
        return st;
    if (out_bytes < (size_t)L.total_bytes)
        return TG_ERR_WORKSPACE;
    uint8_t *out = static_cast<uint8_t *>(out_v);
    std::memset(out, 0, (size_t)L.total_bytes);

    if (kind == TG_TERNARY_I8 || kind == TG_BINARY_Q1) {
        if (!(kind == TG_BINARY_Q1 ? pack_q1(L, trits, out) : pack_masks(L, trits, out)))
            return TG_ERR_VALUE;
        const int64_t G = L.G;
        int64_t maxabs = 0;
        for (int64_t T = 0; T < L.tiles; T++) {
            for (int64_t g = 0; g < G; g++) {
                for (int l = 0; l < tgi::kTileRows; l++) {
                    const int64_t r = T * tgi::kTileRows + l;
                    const int64_t slot = (T * G + g) * tgi::kTileRows + l;
                    int32_t d = r < N ? static_cast<const int32_t *>(scales)[r * G + g] : 0;
                    int64_t a = d < 0 ? -(int64_t)d : (int64_t)d;
                    maxabs = std::max(maxabs, a);
                    store_u32(out + L.scale_off + slot * 4, (uint32_t)d);
                }
            }
        }
        L.max_abs_scale = maxabs;
    } else if (kind == TG_TERNARY_LNS8) {
        if (!pack_lns8_fragments(L, trits, out))
            return TG_ERR_VALUE;
        const int64_t G = L.G;
        int64_t maxc = 0;
        for (int64_t B = 0; B < L.tiles; B++) {
            for (int64_t g = 0; g < G; g++) {
                for (int l = 0; l < tgi::kLnsBlockRows; l++) {
                    const int64_t r = B * tgi::kLnsBlockRows + l;
                    const uint8_t c = r < N ? static_cast<const uint8_t *>(scales)[r * G + g] : 0;
                    maxc = std::max<int64_t>(maxc, c);
                    out[L.scale_off + (B * G + g) * tgi::kLnsBlockRows + l] = c;
                }
            }
        }
        L.max_abs_scale = maxc;
    } else {
        // TG_PLANES8: two balanced base-3 digit groups per weight, W = 81*hi + lo.
        const int32_t *s = static_cast<const int32_t *>(scales);
        int64_t maxs = 0;
        for (int64_t r = 0; r < N; r++) {
            if (s[r] <= 0)
                return TG_ERR_VALUE;
            maxs = std::max<int64_t>(maxs, s[r]);
        }
        const int64_t plane = N * K;
        std::vector<char> bad((size_t)N, 0);
        parallel_rows(N, [&](int64_t r0, int64_t r1) {
            for (int64_t r = r0; r < r1; r++) {
                int m = 0;
                for (int64_t i = 0; i < K; i++) {
                    int hi = 0, lo = 0;
                    for (int p = 0; p < 8; p++) {
                        int8_t v = trits[p * plane + r * K + i];
                        if (v < -1 || v > 1)
                            bad[(size_t)r] = 1;
                        if (p < 4)
                            hi = hi * 3 + v;
                        else
                            lo = lo * 3 + v;
                    }
                    out[L.mask_off + 2 * r * K + i] = (uint8_t)(int8_t)hi;
                    out[L.aux_off + 2 * r * K + i] = (uint8_t)(int8_t)lo;
                    m = std::max(m, lo < 0 ? -lo : lo);
                }
                out[L.aux2_off + r] = (uint8_t)m;
                store_u32(out + L.scale_off + r * 4, (uint32_t)s[r]);
            }
        });
        for (char b : bad)
            if (b)
                return TG_ERR_VALUE;
        L.max_abs_scale = maxs;
    }
    *layout = L;
    return TG_OK;
}
