// Layout of one cached CF-BI row (one token of an open 16-token chunk, one head), shared by the
// token-sequential kernels (cfbi.cu) and the chunk-parallel prefill (cfbi_chunked.cu).
//
// Source: "Kimi K3.1 inference zero mismatch" (LLMNews), section 6.1 (CF-BI): besides the recurrent state,
// the open chunk's rows and its position are kept, so decode continues the chunk with the same row-level
// arithmetic as prefill.
#pragma once
#include "../../include/kda.h"

namespace kda {
namespace cfbi {

constexpr int D = 128;                   // dk = dv
constexpr int CH = KDA_CFBI_CHUNK;       // rows per chunk
constexpr int RF = KDA_CFBI_ROW_FLOATS;  // floats per cached row
// k | v | G (in-chunk cumulative log-decay) | A_t[u] (beta folded in, u < t; zero for u >= t) | beta |
// T_t[v] = row t of (I + A)^-1 (zero for v > t) | zero padding
constexpr int R_K = 0, R_V = 128, R_G = 256, R_A = 384, R_BETA = 400, R_T = 401;
static_assert(R_T + CH <= RF && RF % 4 == 0, "row layout");

}  // namespace cfbi
}  // namespace kda
