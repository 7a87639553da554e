"""The README's usage example runs as written and its selection matches the oracle."""

import os

import numpy as np
import pytest

import parity
import workloads as wl

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_decode_example(orc):
    import torch
    with open(os.path.join(ROOT, "README.md")) as f:
        text = f.read()
    start = text.index("```python") + len("```python")
    code = text[start:text.index("```", start)]
    torch.manual_seed(0)
    env = {}
    exec(compile(code, "README.md", "exec"), env)
    B, L, k = env["B"], env["L"], env["k"]
    w = wl.Workload(name="readme", q=env["q"].cpu().view(torch.int16).numpy().view(np.uint16),
                    pool=env["pool"].cpu().view(torch.int16).numpy().view(np.uint16),
                    block_table=env["block_table"].cpu().numpy(),
                    seq_lens=env["seq_lens"].cpu().numpy(), k=k, n_sink=1, n_window=2,
                    max_model_len=L)
    o_scores, o_ids, _ = orc.run(w)
    parity.check(w, o_scores, o_ids, env["ids"].cpu().numpy(), env["scores"].cpu().numpy())
