"""The Python binding only marshals: every entry point refuses host tensors
(there is no CPU path), a missing library raises instead of falling back, and
the package never reaches the oracle.  No GPU needed."""
import os
import subprocess
import sys

import pytest
import torch

import fmha_block_map_gb300 as fbm
from fmha_block_map_gb300 import cp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _cpu(*shape, dtype=torch.float16):
    return torch.zeros(shape, dtype=dtype)


@pytest.mark.parametrize("call", [
    lambda: fbm.sparge_block_map(_cpu(1, 2, 128, 64), _cpu(1, 2, 128, 64), topk=0.5),
    lambda: fbm.sparse_fmha_fwd(_cpu(1, 2, 128, 64), _cpu(1, 2, 128, 64), _cpu(1, 2, 128, 64),
                                None, None),
    lambda: fbm.attn_combine(_cpu(2, 4, 64, dtype=torch.float32), _cpu(2, 4, dtype=torch.float32)),
    lambda: fbm.lut_shard(_cpu(4, 8, dtype=torch.int32), _cpu(4, dtype=torch.int32), 0, 4),
    lambda: fbm.quantize_e4m3_blocks(_cpu(1, 2, 128, 128)),
    lambda: fbm.sparse_fmha_fwd_fp8(_cpu(1, 2, 128, 128, dtype=torch.uint8),
                                    _cpu(1, 2, 2, dtype=torch.float32),
                                    _cpu(1, 2, 128, 128, dtype=torch.uint8),
                                    _cpu(1, 2, 2, dtype=torch.float32), _cpu(1, 2, 128, 128),
                                    None, None),
    lambda: fbm.sparse_decode_fwd(_cpu(4, 16, 576, dtype=torch.bfloat16),
                                  _cpu(8, 64, 576, dtype=torch.bfloat16),
                                  _cpu(4, 2, dtype=torch.int32), _cpu(4, 32, dtype=torch.int32),
                                  dv=512, scale=0.1),
    lambda: cp.rank_partial(_cpu(1, 2, 128, 128), _cpu(1, 2, 64, 128), _cpu(1, 2, 64, 128),
                            _cpu(1, 2, 2, 2, dtype=torch.int32), _cpu(1, 2, 2, dtype=torch.int32),
                            0, 1),
])
def test_host_tensors_are_refused(call):
    with pytest.raises(ValueError, match="CUDA tensor"):
        call()


def test_missing_library_raises(monkeypatch):
    monkeypatch.setattr(fbm, "_lib", None)
    monkeypatch.setattr(fbm, "LIB_PATH", os.path.join(ROOT, "no_such_dir", "libfbm.so"))
    with pytest.raises(RuntimeError, match="missing"):
        fbm.lib()


def test_package_does_not_reach_the_oracle():
    code = ("import sys; import fmha_block_map_gb300, fmha_block_map_gb300.cp, "
            "fmha_block_map_gb300.build; "
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                         check=True).stdout.strip()
    assert out == "False"
    pkg = os.path.join(ROOT, "fmha_block_map_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "from oracle" not in text, f


def test_kv_shard_bounds_follow_the_chunk_rule():
    import oracle

    for nk in range(1, 40):
        for world in range(1, min(nk, 9) + 1):
            assert cp.kv_shard_bounds(nk, world) == oracle.split_bounds(nk, world)
    for nk, world in ((0, 1), (3, 4), (5, 0)):
        with pytest.raises(ValueError):
            cp.kv_shard_bounds(nk, world)
