// The 16 NormalFloat-4 values as printed in the QLoRA paper (Dettmers et al. 2023, appendix
// "NormalFloat 4-bit data type"); every literal is an exact fp32 value.
#pragma once

#define LM_NF4_VALUES                                                                            \
    -1.0f, -0.6961928009986877f, -0.5250730514526367f, -0.39491748809814453f,                    \
        -0.28444138169288635f, -0.18477343022823334f, -0.09105003625154495f, 0.0f,               \
        0.07958029955625534f, 0.16093020141124725f, 0.24611230194568634f, 0.33791524171829224f,  \
        0.44070982933044434f, 0.5626170039176941f, 0.7229568362236023f, 1.0f

namespace lm {

constexpr float kNf4Values[16] = {LM_NF4_VALUES};

// Value i of the table in host or device code; with a constant index it folds to an immediate.
__host__ __device__ constexpr float nf4_value(int i) {
    constexpr float v[16] = {LM_NF4_VALUES};
    return v[i];
}

}  // namespace lm
