"""The bounded waits of the tcgen05 kernels (the MLA token-split kernel of
the bf16 cache, the MLA kernel of the 8-bit cache, the many-row GQA kernel)
give up after a fixed number of polls, raise DCP_DEVERR_TIMEOUT,
stop every role, drain the copies and MMAs they issued, free tensor memory
and return. This builds a second copy of the library whose poll limit is 1
(-DDCP_SPIN_LIMIT=1), so that each of those kernels aborts at its first wait
that is not already satisfied, and checks, in a fresh process:
  - the call returns and the stream synchronises without a CUDA error;
  - the device error word carries DCP_DEVERR_TIMEOUT;
  - the normal library, called next on the same state in the same process,
    still matches the float64 oracle (the context and the GPU are intact).
No GPU fault or hang is involved: every wait in the kernels is bounded."""
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
pytestmark = pytest.mark.gpu

CHILD = r'''
import sys
sys.path.insert(0, sys.argv[1])
sys.path.insert(0, sys.argv[1] + "/tests")
import numpy as np
import torch
import oracle as O
from helpers import assert_close, assert_lse_close, oracle_mtp_sequence, oracle_sequence
from sequence_sharded_decode_gb300 import configs, dcp
from sequence_sharded_decode_gb300.state import DecodeState

variant, normal = sys.argv[2], sys.argv[3]
cases = [(configs.get("mla_decode").with_(batch=2, ctx_kind="fixed", ctx_fixed=900, shards=3), 1),
         (configs.get("mla_decode").with_(batch=2, ctx_kind="fixed", ctx_fixed=900, shards=3, kv_dtype="fp8"), 1),
         (configs.get("gqa_mid").with_(batch=1, ctx_fixed=700, shards=2), 16)]
for wl, q_len in cases:
    dcp._lib, dcp._LIB_PATH = None, variant
    st = DecodeState(wl, q_len=q_len, gen_device="cpu")
    st.append()                         # the step's new tokens (the append kernel has no waits)
    st.attention()
    torch.cuda.synchronize()            # raises if the kernel faulted
    flag = int(st.err.item())
    assert flag & dcp.DCP_DEVERR_TIMEOUT, f"{wl.name}: expected the timeout bit, flag {flag}"
    assert not flag & ~dcp.DCP_DEVERR_TIMEOUT, f"{wl.name}: unexpected flag bits {flag}"
    dcp._lib, dcp._LIB_PATH = None, normal
    st.err.zero_()
    st.attention()
    torch.cuda.synchronize()
    assert int(st.err.item()) == 0
    o, lse = st.o.cpu().numpy(), st.lse.cpu().numpy()
    for b in range(wl.batch):
        starts_b = O.shard_starts([st.ctx[b]], wl.shards)[0]
        if q_len == 1:
            ro, rl, _, _ = oracle_sequence(wl, b, int(st.ctx[b]) + 1, starts_b)
        else:
            ro, rl, _, _ = oracle_mtp_sequence(wl, b, int(st.ctx[b]), q_len, starts_b)
        assert_close(o[b], ro, f"{wl.name} O[b={b}] after the aborted call")
        assert_lse_close(lse[b], rl, f"{wl.name} LSE[b={b}] after the aborted call")
    print(f"{wl.name}: aborted with DCP_DEVERR_TIMEOUT, then correct")
print("EXPIRY_OK")
'''


def test_wait_expiry_aborts_cleanly(tmp_path):
    from sequence_sharded_decode_gb300 import build, dcp
    variant = build.build(extra=["-DDCP_SPIN_LIMIT=1"], out=str(tmp_path / "libdcp_spin1.so"),
                          build_dir=str(tmp_path / "obj"))
    script = tmp_path / "child.py"
    script.write_text(CHILD)
    r = subprocess.run([sys.executable, str(script), ROOT, variant, dcp.lib_path()], capture_output=True,
                       text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "EXPIRY_OK" in r.stdout
