"""The product path has no CPU fallback: CPU tensors are rejected by the
binding, a missing library raises instead of computing anything, the
package never imports the oracle, and without a GPU the C library returns
an error status rather than computing on the host.  CPU only."""
import ctypes
import os
import subprocess
import sys

import pytest
import torch

import causal_gqa_attention_ne_gb300 as ne

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_cpu_tensors_are_rejected():
    q = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    k = torch.zeros(1, 8, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        ne.attention_forward(q, k, k)


def test_missing_library_raises():
    code = ("import causal_gqa_attention_ne_gb300._build as b; b.LIB = '/nonexistent/libne_attn.so'\n"
            "import causal_gqa_attention_ne_gb300 as ne\n"
            "try:\n"
            "    ne.load_library(build_if_missing=False)\n"
            "except RuntimeError as e:\n"
            "    print('raised', 'missing' in str(e))\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "raised True"


def test_package_never_imports_the_oracle():
    code = ("import sys\n"
            "import causal_gqa_attention_ne_gb300 as ne\n"
            "ne.load_library()\n"
            "print(any(m == 'oracle' or m.startswith('oracle.') for m in sys.modules))\n")
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, capture_output=True, text=True,
                       timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == "False"
    pkg = os.path.join(ROOT, "causal_gqa_attention_ne_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert "import oracle" not in text and "ne_oracle" not in text, f


@pytest.mark.skipif(torch.cuda.is_available(), reason="host pointers must never reach a GPU")
def test_library_without_a_gpu_returns_an_error():
    lib = ne.load_library()
    buf = ctypes.create_string_buffer(1 << 16)
    a = (ctypes.addressof(buf) + 15) // 16 * 16
    rc = lib.ne_attn_fwd(a, a, a, a, a, 1, 8, 2, 2, 64, 10000.0, None)
    assert rc in (3, 6), ne.ne_attn_status_string(rc)      # UNSUPPORTED or CUDA: no host path
