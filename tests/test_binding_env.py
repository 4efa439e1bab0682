"""Importing the binding asks CUDA for 32 hardware work queues unless the caller chose a
number: the library's side and teardown streams then do not share queues with the caller's
streams.  Checked in fresh interpreters, since the variable only matters before the CUDA
context exists."""
import os
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _env_after_import(preset):
    env = {k: v for k, v in os.environ.items() if k != "CUDA_DEVICE_MAX_CONNECTIONS"}
    if preset is not None:
        env["CUDA_DEVICE_MAX_CONNECTIONS"] = preset
    code = ("import os, context_attention_metadata_gb300; "
            "print(os.environ.get('CUDA_DEVICE_MAX_CONNECTIONS'))")
    out = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True,
                         text=True, timeout=120)
    assert out.returncode == 0, out.stderr
    return out.stdout.strip()


def test_import_sets_32_queues_when_unset():
    assert _env_after_import(None) == "32"


def test_import_keeps_the_callers_choice():
    assert _env_after_import("4") == "4"
