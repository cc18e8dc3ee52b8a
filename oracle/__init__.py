"""fp64 CPU oracle of AttnRes residual aggregation.  Test infrastructure only: the product
path never imports this package (see attnres_oracle.py)."""
