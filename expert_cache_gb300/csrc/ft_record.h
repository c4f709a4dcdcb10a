// Byte layout of one expert record (plain C++, shared by the CUDA and the host sources).
#pragma once
#include <stddef.h>

#include "../../include/ft.h"

namespace ft {

struct RecordLayout {
    size_t gu_codes, gu_scales, d_codes, d_scales, s_gu, s_d;
    size_t raw, bytes;
};

// Scale block length along K: 16 (NVFP4, E4M3 scales) or 32 (MXFP4, E8M0 scales).
inline int scale_block(int format) { return format == FT_FORMAT_MXFP4 ? 32 : 16; }

inline RecordLayout record_layout(int H, int I, int format = FT_FORMAT_NVFP4) {
    RecordLayout r;
    const size_t sb = (size_t)scale_block(format);
    size_t off = 0;
    r.gu_codes = off;  off += (size_t)2 * I * H / 2;
    r.gu_scales = off; off += (size_t)2 * I * H / sb;
    r.d_codes = off;   off += (size_t)H * I / 2;
    r.d_scales = off;  off += (size_t)H * I / sb;
    r.s_gu = off;      off += 4;
    r.s_d = off;       off += 4;
    r.raw = off;
    r.bytes = (off + 255) / 256 * 256;
    return r;
}

}  // namespace ft
