"""Optional record of parity margins: when the environment variable
FA_PARITY_LOG names a file, each GPU-versus-oracle comparison appends one
JSON line with its errors, so a run of the GPU tests leaves a table of how
far every case sits from its bound."""
import json
import os


def record(kind: str, what: str, **values) -> None:
    path = os.environ.get("FA_PARITY_LOG")
    if not path:
        return
    with open(path, "a") as f:
        f.write(json.dumps({"kind": kind, "case": what,
                            **{k: float(v) for k, v in values.items()}}) + "\n")
