"""The oracle and its pins run without the library they judge.

The oracle tests are copied, with the oracle, the seeded input generators and
the golden files, into a directory that holds no copy of the library package,
and run there in a fresh interpreter.  A final hook in that run fails if
``libzs.so`` is mapped in the process.  So the oracle side neither imports the
CUDA path nor loads it by a side effect (importing a package whose
``__init__`` opens the library, say).
"""

import glob
import os
import shutil
import subprocess
import sys
import textwrap

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_GUARD = textwrap.dedent('''
    import os
    import sys

    sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))


    def pytest_sessionfinish(session, exitstatus):
        with open("/proc/self/maps") as f:
            mapped = [ln.split()[-1] for ln in f if ln.rstrip().endswith("libzs.so")]
        if mapped:
            session.exitstatus = 9
            print("LIBRARY MAPPED: %s" % sorted(set(mapped)))
''')


_GOLDEN = textwrap.dedent('''

    import pytest


    @pytest.fixture(scope="session")
    def golden_dir():
        return os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
''')


def test_oracle_tests_pass_without_the_library(tmp_path):
    work = tmp_path / "tree"
    tests = work / "tests"
    tests.mkdir(parents=True)
    shutil.copytree(os.path.join(ROOT, "oracle"), work / "oracle",
                    ignore=shutil.ignore_patterns("__pycache__"))
    shutil.copy(os.path.join(ROOT, "synth.py"), work / "synth.py")
    shutil.copytree(os.path.join(ROOT, "tests", "golden"), tests / "golden")
    names = sorted(os.path.basename(p) for p in glob.glob(os.path.join(ROOT, "tests", "test_oracle_*.py")))
    names = [n for n in names if n != os.path.basename(__file__)]
    assert len(names) >= 5, names
    for n in names + ["pins.py"]:
        shutil.copy(os.path.join(ROOT, "tests", n), tests / n)
    # the oracle tests need only the golden-file fixture of the suite's conftest (not its library build)
    (tests / "conftest.py").write_text(_GUARD + _GOLDEN)
    (work / "pytest.ini").write_text("[pytest]\ntestpaths = tests\naddopts = -p no:cacheprovider\n"
                                     "markers =\n    gpu: needs a CUDA GPU\n")
    assert not (work / "fsdp_sharded_optimizer_flatparameter_gb300").exists()
    env = dict(os.environ)
    env.pop("PYTHONPATH", None)
    proc = subprocess.run([sys.executable, "-m", "pytest", "-q", "-m", "not gpu", "-x"], cwd=str(work), env=env,
                          capture_output=True, text=True, timeout=600)
    out = proc.stdout + proc.stderr
    assert proc.returncode == 0, out[-4000:]
    assert "LIBRARY MAPPED" not in out
    assert " passed" in out
