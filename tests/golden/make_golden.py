"""Writes tests/golden/tiny_oracle.json by running only the CPU oracle.

Content: the tiny workload (2 layers, hidden 256, 4 q / 2 kv heads, head_dim 64,
SwiGLU 688, vocab 1024, weights N(0, 0.02) from seed 0) decoded greedily from
its 32-token prompt for 16 steps; the argmax token of every step and the first
logits of a few steps.  It is a regression fixture for the oracle itself (the
same numbers must come out on every host), not a GPU result.

Usage: python tests/golden/make_golden.py
"""
import json
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.dirname(os.path.abspath(__file__))))
sys.path.insert(0, ROOT)

import oracle  # noqa: E402
import synth  # noqa: E402


def run():
    w = synth.WORKLOADS["tiny"]
    m = synth.make_model(w.shape, w.seed_weights)
    prompt = synth.make_prompt(w)
    o = oracle.OracleDecoder(m, w.max_seq())
    tokens, heads = [], {}
    tok = int(prompt[0])
    for p in range(w.prompt_len + w.decode - 1):
        tok = int(prompt[p]) if p < w.prompt_len else tok
        lg, _ = o.step(tok, p)
        nxt, _ = oracle.argmax_f32(lg)
        tokens.append(nxt)
        if p in (0, w.prompt_len - 1, w.prompt_len + w.decode - 2):
            heads[str(p)] = [float(v) for v in lg[:8]]
        tok = nxt
    return {"workload": "tiny", "prompt": [int(t) for t in prompt], "argmax_per_step": tokens,
            "logits_head_at_pos": heads}


if __name__ == "__main__":
    out = os.path.join(os.path.dirname(os.path.abspath(__file__)), "tiny_oracle.json")
    with open(out, "w") as f:
        json.dump(run(), f, indent=1)
    print("wrote", out)
