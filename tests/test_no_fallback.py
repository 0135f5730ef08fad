"""The product path has no CPU fallback: the package never imports the oracle
(or the input generators), and without the native library every call raises
instead of computing anything on the host.  Each case runs in a fresh
interpreter so that the library loaded by the other tests does not mask it."""
import os
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _run(code: str) -> subprocess.CompletedProcess:
    return subprocess.run([sys.executable, "-c", textwrap.dedent(code)], cwd=ROOT, capture_output=True, text=True,
                          timeout=300)


def test_package_does_not_import_the_oracle():
    r = _run("""
        import sys
        import block_causal_masked_gb300 as bd
        bd.lib()
        print("oracle" in sys.modules, "synth" in sys.modules)
    """)
    assert r.returncode == 0, r.stderr
    assert r.stdout.split() == ["False", "False"]


def test_calls_raise_without_the_native_library():
    r = _run("""
        import torch
        import block_causal_masked_gb300 as bd
        from block_causal_masked_gb300 import _build

        def no_toolkit(*args, **kwargs):
            raise RuntimeError("nvcc not found: the CUDA toolkit is required to build libbd")

        _build.build = no_toolkit
        q = torch.zeros((2, 4, 64), dtype=torch.bfloat16)
        kv = torch.zeros((2, 10, 64), dtype=torch.bfloat16)
        try:
            out = bd.bd_block_causal_attn(q, kv, kv, 8, block_size=1)
        except Exception as e:  # any error will do; a result would be a fallback
            print("raised", type(e).__name__)
        else:
            print("returned", type(out).__name__)
    """)
    assert "raised" in r.stdout, r.stdout + r.stderr
