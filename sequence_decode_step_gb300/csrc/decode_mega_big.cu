// The persistent decode kernel built for wide inputs and int4 g128 weights
// (namespace qw::mega_big): 11 consumer warps, an input buffer of 44 x 256 floats
// (the 11008-wide SwiGLU vector of the Qwen2.5-3B shape fits) and five ring
// stages; see decode_mega.cu.
#define QW_MEGA_CONSUMERS 11
#define QW_MEGA_MAXC 44
#define QW_MEGA_STAGES 5
#define QW_MEGA_BIG 1
#define QW_MEGA_NS mega_big
#include "decode_mega.cu"
