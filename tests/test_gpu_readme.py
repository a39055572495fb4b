"""The README's usage example runs as written and matches the float64 oracle."""
import os
import re

import pytest
import torch

import gpu_harness as H
import oracle
import workloads

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_readme_example_matches_the_oracle():
    text = open(os.path.join(ROOT, "README.md")).read()
    code = re.search(r"```python\n(.*?)```", text, re.S).group(1)
    torch.manual_seed(5)
    pool_before = {}
    env = {}
    # run the example up to the fused call, keep the cache as it was, then run the call
    head, call = code.split("vh.vh_decode_fused(", 1)
    exec(head, env)
    pool_before = env["pool"].clone()
    exec("vh.vh_decode_fused(" + call, env)
    torch.cuda.synchronize()
    e = env
    inp = workloads.DecodeInputs(B=e["B"], Hq=e["Hq"], Hkv=e["Hkv"], D=e["D"], P=e["P"], max_pages_per_seq=e["MPS"],
                                 num_pages=e["NP"], theta=10000.0, q=e["q"].cpu(), k_new=e["k_new"].cpu(),
                                 v_new=e["v_new"].cpu(), pool=pool_before.cpu(), page_table=e["page_table"].cpu(),
                                 seq_lens=e["seq_lens"].cpu(), active=e["active"].cpu())
    ref = oracle.reference_step(inp)
    H.check_out(inp, ref["out"], e["out"].cpu())
    H.check_append(inp, ref, e["pool"].cpu())
