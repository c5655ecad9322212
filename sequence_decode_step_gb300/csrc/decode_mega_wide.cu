// The persistent decode kernel built with 11 consumer warps (namespace
// qw::mega_wide), used from long contexts on; see decode_mega.cu.
#define QW_MEGA_CONSUMERS 11
#define QW_MEGA_NS mega_wide
#include "decode_mega.cu"
