"""Free device memory around split calls, measured in a fresh process.

A new Python process is used so that no earlier call of another entry point
has set up the library's split-scratch pool.  In it, a causal call of the
entry point comes first (it needs no scratch; it loads the kernel and sets
the device up), then the free-memory baseline, then ten non-causal calls of
[1,64,2048,128] whose last round is split (on a 152-SM GB300: 112 pieces),
then free memory again.
"""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_SCRIPT = r"""
import math, sys, torch
sys.path.insert(0, {root!r})
import exact_attention_forward_07_gb300 as fa
from attn_inputs import make_qkv
fn = {fn!r}
B, H, N, d = 1, 64, 2048, 128
q, k, v = (x.cuda() for x in make_qkv(B, H, N, d, torch.bfloat16, seed=73))
o = torch.empty_like(q)
lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
def call(causal):
    args = [q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(), B, H, N, d,
            int(causal), 1.0 / math.sqrt(d)]
    if fn != "fa_fwd":
        args += [0, 8.0]
    return getattr(fa.lib(), fn)(*args, None)
assert call(True) == 0
torch.cuda.synchronize()
free0, _ = torch.cuda.mem_get_info()
for _ in range(10):
    assert call(False) == 0
torch.cuda.synchronize()
free1, _ = torch.cuda.mem_get_info()
assert fa.fa_get_status() == 0
print("FREE", free0, free1)
"""


def free_memory_around_split_calls(fn: str):
    """(free bytes before, after) the split calls of entry point `fn`
    (fa_fwd, fa_fwd_ex or fa_fwd_noalloc) in a fresh process."""
    r = subprocess.run([sys.executable, "-c", _SCRIPT.format(root=ROOT, fn=fn)],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    line = [ln for ln in r.stdout.splitlines() if ln.startswith("FREE")][-1]
    _, free0, free1 = line.split()
    return int(free0), int(free1)
