// repack.cu -- host-side conversion of canonical expert records into the
// slot layout the expert kernels read (fragment order, see common.cuh).
// Byte counts are unchanged: a slot matrix holds exactly the canonical bytes
// (plus padding to a 16-byte boundary between matrices when a block-FP8
// scale grid is not a multiple of 16 bytes).
#include <string.h>

#include "common.cuh"

namespace moe {

namespace {

inline uint16_t rd16(const uint8_t* p) { return (uint16_t)(p[0] | (p[1] << 8)); }
inline void wr16(uint8_t* p, uint16_t v) { p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); }
inline void wr32(uint8_t* p, uint32_t v) {
    p[0] = (uint8_t)v; p[1] = (uint8_t)(v >> 8); p[2] = (uint8_t)(v >> 16); p[3] = (uint8_t)(v >> 24);
}

// Q4_0: canonical blocks of 18 bytes; code of (r, c).
struct Q4Src {
    const uint8_t* src;
    int nb;
    uint32_t code(int r, int c) const {
        const uint8_t* blk = src + ((size_t)r * nb + c / 32) * 18;
        const int j = c & 31;
        const uint8_t b = blk[2 + (j & 15)];
        return j < 16 ? (uint32_t)(b & 15) : (uint32_t)(b >> 4);
    }
    uint16_t scale(int r, int b) const { return rd16(src + ((size_t)r * nb + b) * 18); }
};

void repack_q4_0(const uint8_t* src, int R, int C, uint8_t* dst) {
    const int KC = C / 64, RT = R / 16;
    const Q4Src q{src, C / 32};
    uint8_t* codes = dst;
    uint8_t* scales = dst + (size_t)R * C / 2;
    for (int rt = 0; rt < RT; ++rt)
        for (int kc = 0; kc < KC; ++kc) {
            const size_t tile = (size_t)rt * KC + kc;
            for (int lane = 0; lane < 32; ++lane) {
                const int g = lane >> 2, qd = lane & 3;
                const int r0 = rt * 16 + g, r8 = r0 + 8;
                for (int s = 0; s < 4; ++s) {
                    const int c0 = kc * 64 + s * 16 + 2 * qd;
                    const uint32_t w = q.code(r0, c0) | (q.code(r0, c0 + 1) << 16) | (q.code(r8, c0) << 4) |
                                       (q.code(r8, c0 + 1) << 20) | (q.code(r0, c0 + 8) << 8) |
                                       (q.code(r0, c0 + 9) << 24) | (q.code(r8, c0 + 8) << 12) |
                                       (q.code(r8, c0 + 9) << 28);
                    wr32(codes + (tile * 32 + lane) * 16 + s * 4, w);
                }
            }
            for (int g = 0; g < 8; ++g) {
                const int r0 = rt * 16 + g, r8 = r0 + 8;
                uint8_t* p = scales + (tile * 8 + g) * 8;
                wr16(p + 0, q.scale(r0, 2 * kc));
                wr16(p + 2, q.scale(r0, 2 * kc + 1));
                wr16(p + 4, q.scale(r8, 2 * kc));
                wr16(p + 6, q.scale(r8, 2 * kc + 1));
            }
        }
}

void repack_nvfp4(const uint8_t* src, int R, int C, uint8_t* dst) {
    const int KC = C / 64, RT = R / 16;
    const uint8_t* scodes = src;                       // [R][C/2]
    const uint8_t* sscales = src + (size_t)R * C / 2;  // [R][C/16]
    uint8_t* codes = dst;
    uint8_t* scales = dst + (size_t)R * C / 2;
    // e2m1 code of (r, c): low nibble of its byte for even c, high for odd
    auto nib = [&](int r, int c) -> uint32_t {
        const uint8_t v = scodes[(size_t)r * (C / 2) + c / 2];
        return (c & 1) ? (uint32_t)(v >> 4) : (uint32_t)(v & 15);
    };
    auto sc = [&](int r, int b) { return sscales[(size_t)r * (C / 16) + b]; };
    for (int rt = 0; rt < RT; ++rt)
        for (int kc = 0; kc < KC; ++kc) {
            const size_t tile = (size_t)rt * KC + kc;
            for (int lane = 0; lane < 32; ++lane) {
                const int g = lane >> 2, qd = lane & 3;
                const int r0 = rt * 16 + g, r8 = r0 + 8;
                for (int s = 0; s < 4; ++s) {
                    // the Q4_0 word layout: fragment half2 j from the codes at
                    // bits 4j (low half) and 4j + 16 (high half), so one shift
                    // and two masks build its fp16 bits
                    const int c0 = kc * 64 + s * 16 + 2 * qd;
                    const uint32_t w = nib(r0, c0) | (nib(r0, c0 + 1) << 16) | (nib(r8, c0) << 4) |
                                       (nib(r8, c0 + 1) << 20) | (nib(r0, c0 + 8) << 8) | (nib(r0, c0 + 9) << 24) |
                                       (nib(r8, c0 + 8) << 12) | (nib(r8, c0 + 9) << 28);
                    wr32(codes + (tile * 32 + lane) * 16 + s * 4, w);
                }
            }
            for (int g = 0; g < 8; ++g) {
                const int r0 = rt * 16 + g, r8 = r0 + 8;
                uint8_t* p = scales + (tile * 8 + g) * 8;
                for (int s = 0; s < 4; ++s) {
                    p[2 * s] = sc(r0, kc * 4 + s);
                    p[2 * s + 1] = sc(r8, kc * 4 + s);
                }
            }
        }
}

void repack_fp8(const uint8_t* src, int R, int C, uint8_t* dst) {
    const int KC = C / 64, RT = R / 16;
    auto q = [&](int r, int c) { return src[(size_t)r * C + c]; };
    for (int rt = 0; rt < RT; ++rt)
        for (int kc = 0; kc < KC; ++kc) {
            const size_t tile = (size_t)rt * KC + kc;
            for (int lane = 0; lane < 32; ++lane) {
                const int g = lane >> 2, qd = lane & 3;
                const int r0 = rt * 16 + g, r8 = r0 + 8;
                for (int s = 0; s < 4; ++s) {
                    const int c0 = kc * 64 + s * 16 + 2 * qd;
                    uint8_t* p = dst + (tile * 32 + lane) * 32 + s * 8;
                    p[0] = q(r0, c0); p[1] = q(r0, c0 + 1);
                    p[2] = q(r8, c0); p[3] = q(r8, c0 + 1);
                    p[4] = q(r0, c0 + 8); p[5] = q(r0, c0 + 9);
                    p[6] = q(r8, c0 + 8); p[7] = q(r8, c0 + 9);
                }
            }
        }
    const size_t nsc = (size_t)((R + 127) / 128) * ((C + 127) / 128) * 4;
    memcpy(dst + (size_t)R * C, src + (size_t)R * C, nsc);
}

void repack_bf16(const uint8_t* src, int R, int C, uint8_t* dst) {
    const int KC = C / 64, RT = R / 16;
    auto w = [&](int r, int c) -> uint32_t { return rd16(src + ((size_t)r * C + c) * 2); };
    for (int rt = 0; rt < RT; ++rt)
        for (int kc = 0; kc < KC; ++kc) {
            const size_t tile = (size_t)rt * KC + kc;
            for (int lane = 0; lane < 32; ++lane) {
                const int g = lane >> 2, qd = lane & 3;
                const int r0 = rt * 16 + g, r8 = r0 + 8;
                for (int s = 0; s < 4; ++s) {
                    const int c0 = kc * 64 + s * 16 + 2 * qd;
                    uint8_t* p = dst + (tile * 32 + lane) * 64 + s * 16;
                    wr32(p + 0, w(r0, c0) | (w(r0, c0 + 1) << 16));
                    wr32(p + 4, w(r8, c0) | (w(r8, c0 + 1) << 16));
                    wr32(p + 8, w(r0, c0 + 8) | (w(r0, c0 + 9) << 16));
                    wr32(p + 12, w(r8, c0 + 8) | (w(r8, c0 + 9) << 16));
                }
            }
        }
}

void repack_matrix(int fmt, const uint8_t* src, int R, int C, uint8_t* dst) {
    switch (fmt) {
    case FMT_Q4_0: repack_q4_0(src, R, C, dst); break;
    case FMT_NVFP4: repack_nvfp4(src, R, C, dst); break;
    case FMT_FP8_B128: repack_fp8(src, R, C, dst); break;
    default: repack_bf16(src, R, C, dst); break;
    }
}

}  // namespace

// canonical: gate [I x H], up [I x H], down [H x I] (+ 3 fp32 globals for
// NVFP4); slot: the same matrices in fragment order at 16-byte-aligned
// offsets. gscales3 receives the NVFP4 globals (1.0 for other formats).
void repack_record(int fmt, int H, int I, const uint8_t* canonical, uint8_t* slot, float* gscales3) {
    const uint64_t cgu = matrix_bytes(fmt, I, H), cdn = matrix_bytes(fmt, H, I);
    const uint64_t sgu = matrix_stride(fmt, I, H), sdn = matrix_stride(fmt, H, I);
    memset(slot + cgu, 0, sgu - cgu);
    memset(slot + sgu + cgu, 0, sgu - cgu);
    memset(slot + 2 * sgu + cdn, 0, sdn - cdn);
    repack_matrix(fmt, canonical, I, H, slot);
    repack_matrix(fmt, canonical + cgu, I, H, slot + sgu);
    repack_matrix(fmt, canonical + 2 * cgu, H, I, slot + 2 * sgu);
    if (fmt == FMT_NVFP4) {
        memcpy(gscales3, canonical + 2 * cgu + cdn, 12);
    } else {
        gscales3[0] = gscales3[1] = gscales3[2] = 1.0f;
    }
}

}  // namespace moe
