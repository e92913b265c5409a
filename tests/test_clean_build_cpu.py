"""A clean checkout builds: the files git would commit (tracked plus
untracked-but-not-ignored, so no prebuilt library) are copied into a fresh
directory, where __graft_entry__.build() must compile libgdn_b300.so and the
oracle from source and import the package; a second process then imports the
package from that copy alone.  Nothing here needs a GPU."""
import os
import shutil
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _committable_files():
    r = subprocess.run(["git", "ls-files", "--cached", "--others", "--exclude-standard", "-z"],
                       cwd=ROOT, capture_output=True)
    if r.returncode != 0:
        pytest.skip("not a git checkout")
    return [f for f in r.stdout.decode().split("\0") if f and os.path.isfile(os.path.join(ROOT, f))]


def test_build_from_clean_checkout(tmp_path):
    files = _committable_files()
    assert not any(f.endswith(".so") for f in files)
    dst = tmp_path / "repo"
    for f in files:
        os.makedirs(dst / os.path.dirname(f), exist_ok=True)
        shutil.copy2(os.path.join(ROOT, f), dst / f)
    assert not (dst / "gated_deltanet_sequence_prefill_b300" / "libgdn_b300.so").exists()
    env = dict(os.environ, PYTHONDONTWRITEBYTECODE="1")
    code = ("import __graft_entry__ as e; e.build(); "
            "import gated_deltanet_sequence_prefill_b300 as g; print(g.LIB_PATH); print(g.version())")
    r = subprocess.run([sys.executable, "-c", code], cwd=dst, capture_output=True, text=True,
                       env=env, timeout=900)
    assert r.returncode == 0, r.stdout + r.stderr
    lib_path = r.stdout.splitlines()[-2]
    assert lib_path.startswith(str(dst)), lib_path
    assert os.path.exists(lib_path)
    assert (dst / "oracle" / "liboracle.so").exists()
    # a later process imports the built package without rebuilding it
    mtime = os.path.getmtime(lib_path)
    r = subprocess.run([sys.executable, "-c", "import gated_deltanet_sequence_prefill_b300 as g; "
                        "print(g.version())"], cwd=dst, capture_output=True, text=True, env=env,
                       timeout=300)
    assert r.returncode == 0, r.stdout + r.stderr
    assert r.stdout.strip().endswith("sm_103a")
    assert os.path.getmtime(lib_path) == mtime
