"""python -m cross_entropy_loss_ce_gb300 -- build libgbce.so in-tree."""
from .build import build

print(build(force=True))
