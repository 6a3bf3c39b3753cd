"""CPU oracle for the GPT-2 training step (test infrastructure only).

Only the tests, the smoke check and bench.py's CPU-baseline leg may import
this package.  It shares no code with the CUDA library; see oracle/gpt2.py
for what each function computes and the page passage it follows.
"""
from .gpt2 import (  # noqa: F401
    Config, GPT2, GPT2_124M, PARAM_NAMES, DECAYED, param_shapes, num_parameters,
    num_activations, init_params, flatten, unflatten, splitmix64, standard_normal_at,
    encoder_forward, encoder_backward, layernorm_forward, layernorm_backward,
    matmul_forward, matmul_backward, attention_forward, attention_backward,
    gelu_forward, gelu_backward, softmax_forward, crossentropy_forward,
    crossentropy_softmax_backward, adamw_update, lr_schedule, sample_token, generate,
)
