"""Result records of the system runs ("llamacpp-batch-invariance": a verdict is
kept with its evidence).  Each run writes one JSON file: what was run (mode,
seeds, sizes), on what (GPU, git revision, library versions), what was
counted (unique completions per prompt, divergences, the rule-of-three bound
on the divergence rate) and timings.  The file is written to a temporary name
and renamed, so a reader never sees half a record."""
from __future__ import annotations

import json
import os
import subprocess
import time


def _git_sha() -> str | None:
    sha = os.environ.get("BI_GIT_SHA")
    if sha:
        return sha
    try:
        root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
        r = subprocess.run(["git", "rev-parse", "HEAD"], cwd=root, capture_output=True, text=True, timeout=10)
        return r.stdout.strip() or None
    except Exception:
        return None


def environment() -> dict:
    import torch
    env = {"git_sha": _git_sha(), "torch": torch.__version__,
           "time_utc": time.strftime("%Y-%m-%dT%H:%M:%SZ", time.gmtime())}
    if torch.cuda.is_available():
        env["gpu"] = torch.cuda.get_device_name(0)
    return env


def record(name: str, payload: dict, directory: str | None = None) -> str | None:
    """Writes {environment, payload} to <directory>/<name>.json atomically and returns the path; directory
    defaults to $BI_RESULTS_DIR (nothing is written when neither is set)."""
    directory = directory or os.environ.get("BI_RESULTS_DIR")
    if not directory:
        return None
    os.makedirs(directory, exist_ok=True)
    path = os.path.join(directory, f"{name}.json")
    tmp = f"{path}.tmp.{os.getpid()}"
    with open(tmp, "w") as fh:
        json.dump({"name": name, "environment": environment(), "result": payload}, fh, indent=1, sort_keys=True)
        fh.flush()
        os.fsync(fh.fileno())
    os.replace(tmp, path)
    return path
