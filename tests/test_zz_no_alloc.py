"""The allocation-free decode attention entry point (GPU).

llama_op_attention_decode_noalloc serves callers that cannot allocate device
memory when they run attention -- a serving engine whose memory pool already
owns the device, an embedded runtime with a fixed memory budget -- by keeping
its split-KV partials in the library's own fixed-size device array.  Its
output is checked against the fp64 oracle (on every row, or on sampled
sequences for the large case) and against the library's other decode entry
point (llama_op_attention with a caller-provided workspace), over calls made
one after another, which share the array.

This file is collected last so that a run stopping at the first failure has
already run every other test; it loads the library itself, so it also passes
alone in a fresh process.
"""
import numpy as np
import pytest

import oracle
import synth
from _helpers import assert_parity, to_dev, to_f64, torch

pytestmark = pytest.mark.gpu

SCRATCH = 32 << 20
PER_CHUNK_FLOATS = lambda D: D + 2  # o (D values), running max, running sum


def _case(B, start_pos, H, G, D, tag):
    L = start_pos + 3
    q = synth.f32_to_bf16_bits(synth.normal(0, f"noalloc/q{tag}", (B, 1, H, D)))
    kc = synth.f32_to_bf16_bits(synth.normal(0, f"noalloc/k{tag}", (B, G, L, D)))
    vc = synth.f32_to_bf16_bits(synth.normal(0, f"noalloc/v{tag}", (B, G, L, D)))
    return q, kc, vc, L


def _existing(lb, q, kd, vd, L, B, start_pos, H, G, D):
    """Output of the library's other entry point, with a caller-provided workspace."""
    t = torch()
    o = t.empty_like(q)
    n = lb.llama_op_attention_workspace_bytes(lb.LLAMA_BF16, B, 1, start_pos, H, D)
    ws = t.empty(max(n, 16), dtype=t.uint8, device="cuda")
    lb.check(lb.llama_op_attention(lb.LLAMA_BF16, q, lb.make_kv_cache(kd, vd, B, L), o, B, 1, start_pos, H, G, D,
                                   ws, n))
    return o


def _noalloc(lb, qd, kd, vd, L, B, sp, H, G, D):
    t = torch()
    o = t.full_like(qd, float("nan"))
    lb.check(lb.llama_op_attention_decode_noalloc(qd, lb.make_kv_cache(kd, vd, B, L), o, B, sp, H, G, D),
             "llama_op_attention_decode_noalloc")
    t.cuda.synchronize()
    return o


def test_noalloc_decode_matches_the_oracle_and_the_existing_entry_point_on_consecutive_calls():
    import decoder_block_gb300 as lb
    lb.load()
    # calls one after another with different shapes: none may see another
    # call's partials (the array keeps the last call's contents)
    cases = [(8, 1500, 32, 8, 128, "a"),   # 6 chunks of 256 positions
             (3, 700, 9, 3, 64, "b"),      # SmolLM2 grouping, d_head 64
             (200, 100, 9, 3, 64, "c"),    # a single chunk: no partials, o written directly
             (8, 1500, 32, 8, 128, "a")]
    for B, sp, H, G, D, tag in cases:
        q, kc, vc, L = _case(B, sp, H, G, D, tag)
        qd, kd, vd = to_dev(q), to_dev(kc), to_dev(vc)
        got = to_f64(_noalloc(lb, qd, kd, vd, L, B, sp, H, G, D))
        assert np.all(np.isfinite(got))
        what = f"B={B} start_pos={sp} H={H} G={G} D={D}"
        ref = oracle.gqa_attention(synth.as_f64(q), synth.as_f64(kc), synth.as_f64(vc), sp)
        assert_parity(got, ref, "bf16", f"noalloc vs oracle {what}")
        assert_parity(got, to_f64(_existing(lb, qd, kd, vd, L, B, sp, H, G, D)), "bf16",
                      f"noalloc vs existing entry point {what}")


def test_noalloc_batch_that_fills_the_array_then_runs_in_groups():
    """H = 32, D = 128, 4096 cached positions: 16 chunks, 266,240 bytes of
    partials per sequence, so 126 sequences fill the array to within 8 KiB of
    its end; B = 130 runs as a group of 126 and one of 4, the second reusing
    the array.  Sequences at both ends of both groups go through the oracle."""
    import decoder_block_gb300 as lb
    lb.load()
    B, sp, H, G, D = 130, 4095, 32, 4, 128
    per_seq = H * ((sp + 1 + 255) // 256) * PER_CHUNK_FLOATS(D) * 4
    group = SCRATCH // per_seq
    assert group == 126 and SCRATCH - group * per_seq <= 8192
    q, kc, vc, L = _case(B, sp, H, G, D, "full")
    qd, kd, vd = to_dev(q), to_dev(kc), to_dev(vc)
    for _ in range(2):  # two calls in a row
        got = to_f64(_noalloc(lb, qd, kd, vd, L, B, sp, H, G, D))
        assert np.all(np.isfinite(got))
        assert_parity(got, to_f64(_existing(lb, qd, kd, vd, L, B, sp, H, G, D)), "bf16",
                      "noalloc vs existing entry point, B = 130")
        rows = [0, 1, group - 1, group, B - 1]
        ref = oracle.gqa_attention_rows(synth.as_f64(q[rows, 0]), np.arange(len(rows)), [sp] * len(rows),
                                        synth.as_f64(kc[rows]), synth.as_f64(vc[rows]))
        assert_parity(got[rows, 0], ref, "bf16", "noalloc vs oracle, sequences at the group edges")


def test_noalloc_rejects_a_sequence_whose_partials_exceed_its_array():
    import decoder_block_gb300 as lb
    lb.load()
    t = torch()
    H, D = 32, 128
    q = t.zeros((1, H, D), dtype=t.bfloat16, device="cuda")
    kc = t.zeros((1, 8, 16, D), dtype=t.bfloat16, device="cuda")
    kv = lb.make_kv_cache(kc, kc, 1, 600000)  # claims 600000 positions; nothing is launched
    # 2017 chunks of 256 positions: one sequence's partials need more than 32 MiB
    sp = 2016 * 256
    assert H * ((sp + 1 + 255) // 256) * PER_CHUNK_FLOATS(D) * 4 > lb.LLAMA_NOALLOC_SCRATCH_BYTES
    assert lb.llama_op_attention_decode_noalloc(q, kv, q, 1, sp, H, 8, D) == lb.LLAMA_ERR_RANGE
    assert lb.LLAMA_NOALLOC_SCRATCH_BYTES == SCRATCH
