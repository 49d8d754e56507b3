"""CPU oracle for the DeepSeekMoE layer forward (test infrastructure only).

This package is the slow, plain, fp64 statement of what the layer computes,
written from the DeepSeek-V3 Technical Report (DeepSeekMoE paragraph,
auxiliary-loss-free load balancing paragraph, model hyper-parameters
paragraph, fine-grained FP8 quantisation paragraphs and Appendix B.2).

It exists to check the CUDA library, never to stand in for it: only the test
suite, the package's ``smoke()`` entry and the CPU-baseline leg of the
benchmark may import it. It imports nothing from the CUDA package and shares
no code, table or constant with it.
"""

from .moe_oracle import (  # noqa: F401
    sigmoid_affinity,
    biased_scores,
    group_scores,
    select_experts,
    gating_weights,
    expert_load,
    segment_layout,
    permute_rows,
    silu,
    swiglu_ffn,
    combine,
    gate_of_row,
    bias_update,
    moe_layer_forward,
    moe_layer_tokens,
    load_spread,
    sequence_balance,
)
from .fp8 import (  # noqa: F401
    E4M3_MAX,
    e4m3_round,
    e4m3_decode,
    e4m3_encode,
    quantize_act_1x128,
    quantize_weight_128x128,
    dequantize_act_1x128,
    dequantize_weight_128x128,
    fp8_linear,
)
from .moe_fp8 import (  # noqa: F401
    fp8_swiglu_ffn,
    moe_layer_forward_fp8,
    moe_layer_tokens_fp8,
)
from .moe_backward import (  # noqa: F401
    swiglu_ffn_backward,
    gate_backward,
    combine_backward,
    input_grad,
    router_weight_grad,
    moe_layer_backward,
)
from .moe_fp8_backward import (  # noqa: F401
    quantize_act_128x1,
    dequantize_act_128x1,
    fp8_dgrad,
    fp8_wgrad,
    fp8_swiglu_ffn_backward,
)
