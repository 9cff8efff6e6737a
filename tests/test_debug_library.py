"""The debug variant of the library (librar_debug.so, built with RAR_DEBUG:
device-side slice bounds checks) is selected with RAR_LIBRARY=debug, exports
the same entry points and knows the bounds status. CPU only: nothing is
launched."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = r"""
import sys
sys.path.insert(0, {root!r})
from collective_communication_gb300 import binding as B
assert B.library_path().endswith("librar_debug.so"), B.library_path()
L = B.load_library()
for name in B.EXPORTED:
    assert hasattr(L, name), name
assert "debug" in B.strerror(B.Status.ERR_BOUNDS)
print("ok")
"""


def test_debug_library_loads_and_exports_everything():
    from collective_communication_gb300 import build
    build.build(debug=True)
    env = dict(os.environ, RAR_LIBRARY="debug")
    r = subprocess.run([sys.executable, "-c", SCRIPT.format(root=ROOT)], env=env, capture_output=True, text=True,
                       timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == "ok", r.stderr[-2000:]
