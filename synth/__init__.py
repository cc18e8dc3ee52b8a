"""Seeded synthetic inputs shared by the tests, the bench and the oracle runs.  Holds none of
the method's arithmetic: only shapes, distributions and seeds."""
