"""GPU parity of the small-shape latency path (sattn_graph_*): one CUDA graph
launch per step must give the bytes of sattn_prepare + sattn_forward, each
launch must read the inputs' current contents, and the replayed output must
match the oracle within the forward's tolerance."""
import pytest
import torch

import quantized_exact_attention_smoothing_gb300 as sattn
import synth
from helpers import assert_close_output, bf16_bits, to_device_bf16

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("name, overrides", [
    ("c1", {}), ("c2", dict(causal=True)), ("c1", dict(B=2, Hq=4, Hkv=2, Nq=100, Nkv=300, causal=True))])
def test_graph_replay_equals_direct_calls(oracle_mod, name, overrides):
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    w = synth.workload(name, **overrides)
    q, k, v = synth.make_inputs(w, seed=77)
    dq, dk, dv = to_device_bf16(q), to_device_bf16(k), to_device_bf16(v)
    g = sattn.Graph(dq, dk, dv, causal=w.causal)
    try:
        for seed in (78, 79):
            q2, k2, v2 = synth.make_inputs(w, seed=seed)
            dq.copy_(to_device_bf16(q2))
            dk.copy_(to_device_bf16(k2))
            dv.copy_(to_device_bf16(v2))
            out = g.launch()
            assert sattn.check_status(g.workspace) == 0
            got = out.clone()
            ref = sattn.forward(sattn.prepare(dq, dk, dv, w.causal))
            torch.cuda.synchronize()
            assert torch.equal(got.view(torch.int16), ref.view(torch.int16)), f"seed {seed}"
            orc = oracle_mod.prepare(q2, k2, v2)
            rb, _ = oracle_mod.forward(orc, w.Nq, w.Nkv, w.causal)
            assert_close_output(bf16_bits(got), rb, f"graph replay, seed {seed}")
    finally:
        g.close()


def test_graph_as_the_first_call_of_a_process(tmp_path):
    # a fresh process whose first library call is sattn_graph_create: the
    # helper streams and kernel attributes are set up before the capture
    import os
    import subprocess
    import sys
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    script = tmp_path / "graph_first.py"
    script.write_text(
        "import sys, torch\n"
        f"sys.path.insert(0, {root!r}); sys.path.insert(0, {os.path.join(root, 'tests')!r})\n"
        "import synth, quantized_exact_attention_smoothing_gb300 as sattn\n"
        "from helpers import assert_close_output, bf16_bits, to_device_bf16\n"
        "w = synth.workload('c1', causal=True)\n"
        "q, k, v = (to_device_bf16(x) for x in synth.make_inputs(w, seed=5))\n"
        "g = sattn.Graph(q, k, v, causal=True)\n"
        "got = g.launch().clone()\n"
        "assert sattn.check_status(g.workspace) == 0\n"
        "ref = sattn.forward(sattn.prepare(q, k, v, True))\n"
        "torch.cuda.synchronize()\n"
        "assert torch.equal(got.view(torch.int16), ref.view(torch.int16))\n"
        "g.close()\n"
        "print('ok')\n")
    r = subprocess.run([sys.executable, str(script)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), r.stdout + r.stderr
