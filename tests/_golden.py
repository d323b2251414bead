"""Reader for the text fixtures under tests/golden/ ('#' comments, 'key: values' lines)."""
from pathlib import Path

GOLDEN = Path(__file__).resolve().parent / "golden"


def load(name: str) -> dict[str, str]:
    out: dict[str, str] = {}
    for line in (GOLDEN / name).read_text(encoding="utf-8").splitlines():
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        k, _, v = line.partition(":")
        out[k.strip()] = v.strip()
    return out


def nums(s: str, cast=float) -> list:
    return [cast(t) for t in s.replace(",", " ").split()]
