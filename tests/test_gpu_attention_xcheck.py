"""The tcgen05 attention kernel against the warp-level mma.sync kernel: two
independent GPU implementations of the same attention, on the same inputs."""

import os
import subprocess
import sys

import numpy as np
import pytest

from parity import assert_parity, bf16_to_f64

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys, numpy as np, torch
sys.path.insert(0, {root!r})
from dense_decoder_layer_gb300 import pds
B, s, H, Hkv, hd = {shape}
g = torch.Generator().manual_seed(B + s)
q = (torch.randn(B, H, hd, generator=g)).to(torch.bfloat16).cuda()
k = (torch.randn(s + B, Hkv, hd, generator=g)).to(torch.bfloat16).cuda()
v = (torch.randn(s + B, Hkv, hd, generator=g)).to(torch.bfloat16).cuda()
o = torch.empty(B, H * hd, dtype=torch.bfloat16, device="cuda")
pds.pds_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), B, s, H, Hkv, hd,
                  torch.cuda.current_stream().cuda_stream)
torch.cuda.synchronize()
np.save({out!r}, o.view(torch.int16).cpu().numpy())
"""


def _run(shape, mode, tmp_path):
    out = str(tmp_path / f"o_{mode}.npy")
    env = dict(os.environ)
    env.pop("PDS_ATTN", None)
    if mode == "mma":
        env["PDS_ATTN"] = "mma"
    subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT, shape=shape, out=out)],
                   check=True, env=env, timeout=300)
    bits = np.load(out)
    return bf16_to_f64(torch.from_numpy(bits).view(torch.bfloat16))


@pytest.mark.parametrize("shape", [(512, 1536, 24, 8, 128), (300, 77, 8, 2, 64)])
def test_tcgen05_attention_matches_mma_kernel(shape, tmp_path):
    a = _run(shape, "tc", tmp_path)
    b = _run(shape, "mma", tmp_path)
    assert_parity(a, b, f"tcgen05 vs mma.sync attention {shape}")
