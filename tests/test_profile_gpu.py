"""Per-step tracing of a block forward (llama_block_profile_*), GPU.

Each step that launches a kernel of its own is timed once per forward; steps
fused into another step's kernel (RoPE + KV write in the QKV epilogue,
ffn_norm in the O and gate/up epilogues of a bf16 block with d_head 64) read
zero launches.
"""
import pytest

import synth
from _helpers import GpuBlock, to_dev, torch

pytestmark = pytest.mark.gpu


def test_profile_counts_only_steps_that_launch_a_kernel():
    import decoder_block_gb300 as lb
    lb.load()
    t = torch()
    s = dict(synth.SHAPES["smollm2_135m"], max_seq_len=64)
    B, S, n = 2, 64, 3
    with GpuBlock(s, synth.block_weights(s), B * S) as blk:
        x = to_dev(synth.block_activations(s, B=B, S=S))
        y = t.empty_like(x)
        kc, vc = synth.kv_cache(s, max_batch=B, max_seq_len=S)
        kd, vd = to_dev(kc), to_dev(vc)
        lb.check(lb.llama_block_profile_enable(blk.h, n))
        for _ in range(n):
            lb.check(blk.forward(x, y, B, S, 0, kd, vd))
        st, launches, total_ms = lb.llama_block_profile_read(blk.h)
        lb.check(st)
        lb.check(lb.llama_block_profile_disable(blk.h))
    names = [lb.llama_profile_step_name(i) for i in range(lb.LLAMA_PROFILE_STEPS)]
    fused = {2, 5}  # RoPE + KV write, ffn_norm
    for i in range(lb.LLAMA_PROFILE_STEPS):
        if i in fused:
            assert launches[i] == 0 and total_ms[i] == 0.0, names[i]
        else:
            assert launches[i] == n and total_ms[i] > 0.0, names[i]
